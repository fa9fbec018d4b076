"""Bounded waits of the tensor-core kernels, run out on purpose without a GPU
fault: the test hook rswa_debug_set_wait_limit_ns shortens the bound on each
wait for a pipeline phase to 1 ns, so the first phase that is not complete
when first polled gives up.  The kernel then drains its own copies and
tensor-core work (those waits keep their one-second bound), frees its tensor
memory and sets the device flag: rswa_sync_status reports RSWA_EDEVICE, the
context stays usable, and the next call with the default bound is correct
(checked against the oracle)."""

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

RSWA_EDEVICE = 6
BF16_MAX, BF16_MEAN = 2e-2, 5e-3


def f64(t):
    return t.detach().double().cpu().numpy()


def _close(got, ref, what):
    err = np.abs(np.asarray(got, dtype=np.float64) - ref)
    assert np.isfinite(err).all(), what
    assert err.max() <= BF16_MAX and err.mean() <= BF16_MEAN, \
        f"{what}: max {err.max():.3e} mean {err.mean():.3e}"


def _timed_out(rswa, cache, run):
    rswa.rswa_debug_set_wait_limit_ns(1)
    try:
        run()
    finally:
        rswa.rswa_debug_set_wait_limit_ns(0)
    return cache.sync_status()


# (m, T): short units run the persistent prefill, long ones one unit per CTA
@pytest.mark.parametrize("m,T", [(300, 200), (6000, 0)])
def test_prefill_wait_runs_out_then_recovers(cuda_lib, m, T):
    rswa = cuda_lib
    H, d, n = 2, 128, 128
    Q, K, V = (x.cuda() for x in workloads.qkv(m + T, H, d, seed=51))
    cache = rswa.RswaCache(m, n, H, d, 1, rswa.RSWA_BF16)
    O = torch.empty_like(Q)
    status = _timed_out(rswa, cache, lambda: cache.prefill(Q, K, V, O, [m], T))
    assert status == RSWA_EDEVICE
    assert cache.sync_status() == 0                     # the flag was cleared
    O.fill_(float("nan"))
    cache.prefill(Q, K, V, O, [m], T)
    torch.cuda.synchronize()
    assert cache.sync_status() == 0
    rows = sorted({0, 127, 128, m - 1, m, m + T - 1, (m + T) // 2} & set(range(m + T)))
    ref, _ = oracle.prefill_attention(f64(Q), f64(K), f64(V), m, n, rows)
    _close(f64(O[rows]), ref, "prefill after the timeout")


def test_block_wait_runs_out_then_recovers(cuda_lib):
    rswa = cuda_lib
    H, d, n, m, C = 4, 128, 128, 288, 64
    T = 2 * C
    Q, K, V = workloads.qkv(m + T, H, d, seed=52)
    cache = rswa.RswaCache(m, n, H, d, 1, rswa.RSWA_BF16)
    cache.prefill(None, K[:m].cuda(), V[:m].cuda(), None, [m], 0)
    blk = [tuple(x[m + i * C:m + (i + 1) * C][None].contiguous().cuda()
                 for x in (Q, K, V)) for i in range(2)]
    o = torch.empty_like(blk[0][0])
    status = _timed_out(rswa, cache, lambda: cache.decode_block(*blk[0], o))
    assert status == RSWA_EDEVICE
    assert cache.get_t(0) == C                          # the append still ran
    cache.decode_block(*blk[1], o)
    torch.cuda.synchronize()
    assert cache.sync_status() == 0
    ref, _ = oracle.prefill_attention(f64(Q), f64(K), f64(V), m, n,
                                      range(m + C, m + 2 * C))
    _close(f64(o[0]), ref, "block after the timeout")
    assert cache.get_t(0) == 2 * C


@pytest.mark.parametrize("m,H,Hkv,B", [(10272, 10, 10, 1),      # streaming decode
                                       (1400, 16, 4, 24),       # grouped, stream-K
                                       (1400, 32, 2, 24)])      # grouped, one CTA per chunk
def test_decode_wait_runs_out_then_recovers(cuda_lib, m, H, Hkv, B):
    """A fused decode step whose phase waits run out reports RSWA_EDEVICE and
    still appends its key and value; after the documented recovery
    (rswa_cache_set_t with the intended t_b, which also clears the split-K
    counters) the next step, with the default bound, matches the oracle."""
    rswa = cuda_lib
    d, n = 128, 128
    K = workloads.normal((B * m, Hkv, d), 61, 1.0, torch.bfloat16)
    V = workloads.normal((B * m, Hkv, d), 62, 1.0, torch.bfloat16)
    cache = rswa.RswaCache(m, n, H, d, B, rswa.RSWA_BF16, kv_heads=Hkv)
    cache.prefill(None, K.cuda(), V.cuda(), None, [m] * B, 0)
    states = [oracle.prefill_cache(f64(K[b * m:(b + 1) * m]), f64(V[b * m:(b + 1) * m]),
                                   m, n, 0) for b in range(B)]
    steps = [tuple(workloads.normal((B, h, d), 63 + 3 * s + i, 1.0, torch.bfloat16).cuda()
                   for i, h in enumerate((H, Hkv, Hkv))) for s in range(2)]
    o = torch.empty(B, H, d, dtype=torch.bfloat16, device="cuda")
    status = _timed_out(rswa, cache, lambda: cache.decode_step_fused(*steps[0], o))
    assert status == RSWA_EDEVICE
    cache.set_t([1] * B)
    cache.decode_step_fused(*steps[1], o)
    torch.cuda.synchronize()
    assert cache.sync_status() == 0
    for b in range(B):
        for s in range(2):
            q, k, v = (f64(x[b]) for x in steps[s])
            states[b], ro, _ = oracle.decode_step_fused(states[b], q, k, v, n)
        _close(f64(o[b]), ro, f"seq {b} after the timeout")
        assert cache.get_t(b) == 2
