"""rswa_decode_step_fused_static: the fused decode step for callers that must
not allocate device memory once decoding runs (a fixed buffer budget, or a
host application that owns every device byte).  Its split-K scratch comes from
a fixed 4 MiB array inside the library instead of the cache buffer.

Checked through the C ABI against rswa_decode_step_fused on two caches with
identical contents, over two calls in a row, at the bf16 tolerances the other
parity tests use.  This file is collected last on purpose."""

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN = 2e-2, 5e-3


def _two_caches(rswa, m_list, n, H, d, seed, Hkv=None):
    B = len(m_list)
    rows = sum(m_list)
    Hkv = H if Hkv is None else Hkv
    K = workloads.normal((rows, Hkv, d), 3 * seed + 1, 1.0, torch.bfloat16, "cuda")
    V = workloads.normal((rows, Hkv, d), 3 * seed + 2, 1.0, torch.bfloat16, "cuda")
    caches = []
    for _ in range(2):
        c = rswa.RswaCache(max(m_list), n, H, d, B, rswa.RSWA_BF16, kv_heads=Hkv)
        c.prefill(None, K, V, None, m_list, 0)
        caches.append(c)
    return caches


@pytest.mark.parametrize("m_list,n,Hkv", [([288], 128, 4), ([300, 17, 1029], 16, 4),
                                          ([300, 17, 1029], 16, 1)])
def test_static_scratch_matches_fused(cuda_lib, m_list, n, Hkv):
    # Hkv = 1: four query heads over one KV head (the grouped decode path).
    rswa = cuda_lib
    H, d = 4, 128
    B = len(m_list)
    ref_cache, static_cache = _two_caches(rswa, m_list, n, H, d, seed=3, Hkv=Hkv)
    q_all = workloads.normal((2 * B, H, d), 132, 1.0, torch.bfloat16, "cuda")
    k_all = workloads.normal((2 * B, Hkv, d), 133, 1.0, torch.bfloat16, "cuda")
    v_all = workloads.normal((2 * B, Hkv, d), 134, 1.0, torch.bfloat16, "cuda")
    steps = (q_all, k_all, v_all)
    for call in range(2):
        q, k, v = (x[call * B:(call + 1) * B].contiguous() for x in steps)
        o_ref = torch.empty(B, H, d, dtype=torch.bfloat16, device="cuda")
        o_new = torch.full_like(o_ref, float("nan"))
        l_ref = torch.empty(B, H, device="cuda")
        l_new = torch.full_like(l_ref, float("nan"))
        rswa.rswa_decode_step_fused(ref_cache.handle, q, k, v, o_ref, l_ref)
        rswa.rswa_decode_step_fused_static(static_cache.handle, q, k, v, o_new,
                                           l_new)
        torch.cuda.synchronize()
        err = (o_new.double() - o_ref.double()).abs()
        assert torch.isfinite(err).all()
        assert err.max().item() <= BF16_MAX and err.mean().item() <= BF16_MEAN
        assert (l_new - l_ref).abs().max().item() <= 1e-3
        for b in range(B):
            assert static_cache.get_t(b) == ref_cache.get_t(b) == call + 1
    assert static_cache.sync_status() == 0
    # both caches hold the same prefix and the same two ring slots
    Kr, Vr = ref_cache.slabs()
    Ks, Vs = static_cache.slabs()
    m_cap = max(m_list)
    for b, m in enumerate(m_list):
        for A, C in ((Kr, Ks), (Vr, Vs)):
            assert torch.equal(A[b, :, :m], C[b, :, :m])
            assert torch.equal(A[b, :, m_cap:m_cap + 2], C[b, :, m_cap:m_cap + 2])


def test_static_scratch_rejects_oversize(cuda_lib):
    rswa = cuda_lib
    # 1024 sequences x 8 heads x 2 chunks x 66 floats: > 4 MiB of scratch
    cache = rswa.RswaCache(64, 64, 8, 64, 1024, rswa.RSWA_F32)
    q = torch.zeros(1024, 8, 64, device="cuda")
    o = torch.empty_like(q)
    with pytest.raises(rswa.RswaError) as e:
        rswa.rswa_decode_step_fused_static(cache.handle, q, q, q, o)
    assert e.value.status == 2
    assert cache.get_t(0) == 0        # nothing ran
