"""rswa_decode_step_fused_static: the fused decode step for callers that must
not allocate device memory once decoding runs - a serving loop with a fixed
buffer budget (cudaMalloc can stall the device while it synchronises, and
can fail when memory is fragmented), or a plug-in whose host application owns
every device byte.  The call takes its split-K scratch from a fixed 4 MiB
array inside the library instead of the cache buffer.

Each case runs two calls in a row through the C ABI and checks the output,
lse, t_b and the ring against rswa_decode_step_fused on an identical cache
and against the CPU float64 oracle, at the bf16 tolerances of the other
parity tests (max |err| <= 2e-2, mean |err| <= 5e-3).  The cases take the
decode paths that use scratch: split-K, the shared-memory streaming kernel
and the grouped-head tensor-core kernel.  This file is collected last on
purpose."""

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN = 2e-2, 5e-3


def f64(t):
    return t.detach().double().cpu().numpy()


def _close(got, ref, what):
    err = np.abs(np.asarray(got, dtype=np.float64) - ref)
    assert np.isfinite(err).all(), what
    assert err.max() <= BF16_MAX, f"{what}: max {err.max():.3e}"
    assert err.mean() <= BF16_MEAN, f"{what}: mean {err.mean():.3e}"


CASES = [
    # (m_list, n, H, Hkv): the path each shape takes on a 152-SM GB300
    ([2000], 128, 10, 10),            # one sequence, split-K (10.9 MB per step)
    ([300, 17, 1029], 16, 4, 4),      # ragged prefixes, split-K
    ([10272], 128, 10, 10),           # 40-page prefix: the streaming kernel
    ([300, 17, 1029], 16, 4, 1),      # 4 query heads per KV head: tensor cores
]


@pytest.mark.parametrize("m_list,n,H,Hkv", CASES,
                         ids=lambda c: str(c).replace(" ", ""))
def test_static_scratch_matches_fused_and_oracle(cuda_lib, m_list, n, H, Hkv):
    rswa = cuda_lib
    d, seed = 128, 3
    B = len(m_list)
    rows = sum(m_list)
    K = workloads.normal((rows, Hkv, d), 3 * seed + 1, 1.0, torch.bfloat16)
    V = workloads.normal((rows, Hkv, d), 3 * seed + 2, 1.0, torch.bfloat16)
    ref_cache, static_cache = (rswa.RswaCache(max(m_list), n, H, d, B, rswa.RSWA_BF16,
                                              kv_heads=Hkv) for _ in range(2))
    for c in (ref_cache, static_cache):
        c.prefill(None, K.cuda(), V.cuda(), None, m_list, 0)
    offs = np.cumsum([0] + list(m_list))
    states = [oracle.prefill_cache(f64(K[offs[b]:offs[b + 1]]),
                                   f64(V[offs[b]:offs[b + 1]]), m_list[b], n, 0)
              for b in range(B)]
    q_all = workloads.normal((2 * B, H, d), 132, 1.0, torch.bfloat16, "cuda")
    k_all = workloads.normal((2 * B, Hkv, d), 133, 1.0, torch.bfloat16, "cuda")
    v_all = workloads.normal((2 * B, Hkv, d), 134, 1.0, torch.bfloat16, "cuda")
    for call in range(2):
        q, k, v = (x[call * B:(call + 1) * B].contiguous() for x in (q_all, k_all, v_all))
        o_ref = torch.empty(B, H, d, dtype=torch.bfloat16, device="cuda")
        o_new = torch.full_like(o_ref, float("nan"))
        l_ref = torch.empty(B, H, device="cuda")
        l_new = torch.full_like(l_ref, float("nan"))
        rswa.rswa_decode_step_fused(ref_cache.handle, q, k, v, o_ref, l_ref)
        rswa.rswa_decode_step_fused_static(static_cache.handle, q, k, v, o_new, l_new)
        torch.cuda.synchronize()
        _close(f64(o_new), f64(o_ref), f"call {call}: against rswa_decode_step_fused")
        assert (l_new - l_ref).abs().max().item() <= 1e-3
        for b in range(B):
            states[b], ro, rl = oracle.decode_step_fused(
                states[b], f64(q[b]), f64(k[b]), f64(v[b]), n)
            _close(f64(o_new[b]), ro, f"call {call} seq {b}: against the oracle")
            assert np.abs(f64(l_new[b]) - rl).max() <= 1e-3
            assert static_cache.get_t(b) == ref_cache.get_t(b) == call + 1
    assert static_cache.sync_status() == 0
    # the same prefix and ring slots as the oracle's state
    Ks, Vs = static_cache.slabs()
    m_cap = max(m_list)
    for b, m in enumerate(m_list):
        np.testing.assert_array_equal(f64(Ks[b, :, :m]).transpose(1, 0, 2),
                                      states[b]["Kp"])
        np.testing.assert_array_equal(f64(Ks[b, :, m_cap:m_cap + 2]).transpose(1, 0, 2),
                                      states[b]["Kr"][:2])
        np.testing.assert_array_equal(f64(Vs[b, :, m_cap:m_cap + 2]).transpose(1, 0, 2),
                                      states[b]["Vr"][:2])


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
