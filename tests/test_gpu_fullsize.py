"""Parity at the benchmark's full sizes, in the launch configuration that
bench.py times, on outputs the oracle computes one by one."""

import numpy as np
import pytest
import torch

import bench
import oracle

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN = 2e-2, 5e-3


def f64(t):
    return t.detach().double().cpu().numpy()


def check(got, ref, what):
    err = np.abs(np.asarray(got, np.float64) - ref)
    assert np.isfinite(err).all(), what
    assert err.max() <= BF16_MAX, f"{what}: max {err.max():.3e}"
    assert err.mean() <= BF16_MEAN, f"{what}: mean {err.mean():.3e}"


def test_single_page_graph_replay(cuda_lib):
    dev = torch.device("cuda", 0)
    sp = bench.setup_single_page(dev)
    w = sp["w"]
    m, n, T = w.m, w.n, w.T
    s = sp["stream"]
    with torch.cuda.stream(s):
        sp["g_prefill"].replay()
        sp["g_decode"].replay()
    torch.cuda.synchronize()
    # replay once more: every step restarts from an empty ring
    with torch.cuda.stream(s):
        sp["g_prefill"].replay()
        sp["g_decode"].replay()
    torch.cuda.synchronize()
    assert sp["cache"].sync_status() == 0
    Q, K, V = f64(sp["Q"]), f64(sp["K"]), f64(sp["V"])
    ts = [0, 1, 2, 126, 127, 128, 129, 255, 1000, 4097, T - 1]
    ref, _ = oracle.prefill_attention(Q, K, V, m, n, rows=[m + t for t in ts])
    check(f64(sp["Od"][ts, 0]), ref, "decode rows")
    pr = [0, 1, 100, 127, 128, m - 1]
    refp, _ = oracle.prefill_attention(Q, K, V, m, n, rows=pr)
    check(f64(sp["Op"][pr]), refp, "prefix rows")
    assert sp["cache"].get_t(0) == T
    assert sp["cache"].cache_bytes(0) == oracle.cache_len(m, n, T) * 10 * 128 * 2 * 2


def _seq_state(K, V, off, m, n, T):
    return oracle.prefill_cache(f64(K[off:off + m + T]), f64(V[off:off + m + T]),
                                m, n, T)


def test_batched_decode_full(cuda_lib):
    dev = torch.device("cuda", 0)
    bt = bench.setup_batched(dev)
    w = bt["w"]
    B, H, d, n, T = w.batch, w.heads, w.head_dim, w.n, w.T
    q, k, v = (x[:B] for x in bt["steps"])
    o = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, H, device=dev)
    bt["cache"].decode_step_fused(q, k, v, o, lse)
    torch.cuda.synchronize()
    assert bt["cache"].sync_status() == 0
    offs = np.cumsum([0] + [m + T for m in bt["m_list"]])
    for b in [0, 1, 17, 33, 63]:
        m = bt["m_list"][b]
        st = _seq_state(bt["K"], bt["V"], offs[b], m, n, T)
        st, ro, rl = oracle.decode_step_fused(st, f64(q[b]), f64(k[b]), f64(v[b]), n)
        check(f64(o[b]), ro, f"seq {b} (m={m})")
        assert np.abs(f64(lse[b]) - rl).max() <= 1e-3
        assert bt["cache"].get_t(b) == T + 1
        assert bt["cache"].cache_len(b) == oracle.cache_len(m, n, T + 1)


def test_batched_gqa_decode_full(cuda_lib):
    """The batched GQA extra (B 64, H 32 over 8 KV heads, m ~ U{256..2048},
    ring full) in bench.py's launch configuration, sampled sequences."""
    dev = torch.device("cuda", 0)
    gq = bench.setup_batched_gqa(dev)
    w = gq["w"]
    B, d, n, T, H = w.batch, w.head_dim, w.n, w.T, gq["H"]
    q, k, v = (x[:B] for x in gq["steps"])
    o = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, H, device=dev)
    gq["cache"].decode_step_fused(q, k, v, o, lse)
    torch.cuda.synchronize()
    assert gq["cache"].sync_status() == 0
    offs = np.cumsum([0] + [m + T for m in gq["m_list"]])
    for b in [0, 7, 31, 63]:
        m = gq["m_list"][b]
        st = _seq_state(gq["K"], gq["V"], offs[b], m, n, T)
        st, ro, rl = oracle.decode_step_fused(st, f64(q[b]), f64(k[b]), f64(v[b]), n)
        check(f64(o[b]), ro, f"seq {b} (m={m})")
        assert np.abs(f64(lse[b]) - rl).max() <= 1e-3
        assert gq["cache"].get_t(b) == T + 1


@pytest.mark.parametrize("T", [256, 100000])
def test_sweep_decode_full(cuda_lib, T):
    dev = torch.device("cuda", 0)
    sw = bench.setup_sweep(dev)
    w = sw["w"]
    B, H, d, m, n = w.batch, w.heads, w.head_dim, w.m, w.n
    sw["cache"].set_t([T] * B)
    q, k, v = (x[:B] for x in sw["steps"])
    o = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)
    sw["cache"].decode_step_fused(q, k, v, o)
    torch.cuda.synchronize()
    for b in [0, 13, 31]:
        st = _seq_state(sw["K"], sw["V"], b * (m + n), m, n, n)
        st["t"] = T
        st, ro, _ = oracle.decode_step_fused(st, f64(q[b]), f64(k[b]), f64(v[b]), n)
        check(f64(o[b]), ro, f"T={T} seq {b}")
    Ks, _ = sw["cache"].slabs()
    np.testing.assert_array_equal(f64(Ks[5, :, m + T % n]), f64(k[5]))


def test_multipage_prefill_full(cuda_lib):
    dev = torch.device("cuda", 0)
    pf = bench.setup_prefill(dev, layers=1)
    w = pf["w"]
    m, n, T = w.m, w.n, w.T
    L = m + T
    (Q, K, V), cache, O = pf["qkv"][0], pf["caches"][0], pf["outs"][0]
    cache.prefill(Q, K, V, O, [m], T)
    torch.cuda.synchronize()
    assert cache.sync_status() == 0
    rng = np.random.default_rng(0)
    rows = sorted(set([0, 1, 127, 128, 129, 4095, m - 1, m, m + 1, m + 96,
                       m + 127, m + 128, m + 129, 16383, 16384, L - 129, L - 1]
                      + rng.integers(0, L, 16).tolist()))
    ref, _ = oracle.prefill_attention(f64(Q), f64(K), f64(V), m, n, rows=rows)
    check(f64(O[rows]), ref, "multipage rows")
    assert cache.get_t(0) == T
    assert cache.cache_len(0) == m + n
