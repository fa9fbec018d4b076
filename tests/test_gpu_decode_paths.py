"""GPU parity of the decode paths chosen by shape, against the CPU float64
oracle through the C ABI.

* Few heads with long caches: the shared-memory streaming kernel
  (decode_stream.cu), S CTAs per head over [prefix | ring].  Ragged prefixes,
  an empty prefix, a ring that wraps, float32 and head_dim 64, grouped heads
  that no grouped kernel takes, fused and unfused steps enqueued back to
  back (the launches after the first read prefix rows before their
  dependency wait), and the 40-page single-sequence shape.
* Grouped heads on the tensor cores, several fused steps back to back at a
  batched shape whose grid takes more than one wave of CTAs.

Tolerances as in test_gpu_parity: float32 max |err| <= 1e-4; bf16 max |err|
<= 2e-2 and mean |err| <= 5e-3; t_b and cache sizes bit-exact.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

F32_TOL = 1e-4
BF16_MAX, BF16_MEAN = 2e-2, 5e-3


def f64(t):
    return t.detach().double().cpu().numpy()


def assert_close(got, ref, dtype, what=""):
    err = np.abs(np.asarray(got, dtype=np.float64) - ref)
    assert np.isfinite(err).all(), what
    if dtype == 0:
        assert err.max() <= F32_TOL, f"{what}: max {err.max():.3e}"
    else:
        assert err.max() <= BF16_MAX, f"{what}: max {err.max():.3e}"
        assert err.mean() <= BF16_MEAN, f"{what}: mean {err.mean():.3e}"


def tdt(dtype):
    return torch.float32 if dtype == 0 else torch.bfloat16


# Each case moves at least 96 KB of keys and values per SM of a 152-SM GB300
# (the streaming kernel's threshold); the last two are below it and check
# the split-K fallback of the same shapes.
STREAM_CASES = [
    # (m_list, n, H, Hkv, d, dtype, steps, t0)  t0: restored t_b (None: 0)
    ([3000, 1200, 0], 64, 4, 4, 128, 1, 150, None),
    ([9000], 128, 4, 4, 64, 0, 40, None),
    ([4000], 64, 4, 4, 128, 0, 70, None),
    ([14000], 256, 5, 5, 64, 1, 20, 4096 + 37),
    ([1700, 640], 16, 6, 2, 128, 0, 35, None),   # 3 query heads per KV head
    ([10272], 128, 10, 10, 128, 1, 3, 4096 + 37),  # one sequence, 40 pages
    ([2000], 128, 3, 3, 64, 0, 40, None),
    ([900], 32, 2, 2, 128, 0, 70, None),
]


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("case", STREAM_CASES,
                         ids=lambda c: f"m{c[0]}n{c[1]}H{c[2]}kv{c[3]}d{c[4]}dt{c[5]}")
def test_stream_decode(cuda_lib, case, fused):
    rswa = cuda_lib
    m_list, n, H, Hkv, d, dtype, steps, t0 = case
    B = len(m_list)
    dt = tdt(dtype)
    T = n if t0 is not None else 0           # outputs prefilled into the ring
    rows = [m + T for m in m_list]
    K = workloads.normal((sum(rows), Hkv, d), 301, 1.0, dt)
    V = workloads.normal((sum(rows), Hkv, d), 302, 1.0, dt)
    cache = rswa.RswaCache(max(m_list), n, H, d, B, dtype, kv_heads=Hkv)
    cache.prefill(None, K.cuda(), V.cuda(), None, m_list, T)
    offs = np.cumsum([0] + rows)
    states = [oracle.prefill_cache(f64(K[offs[b]:offs[b + 1]]),
                                   f64(V[offs[b]:offs[b + 1]]), m_list[b], n, T)
              for b in range(B)]
    if t0 is not None:
        cache.set_t([t0] * B)
        for st in states:
            st["t"] = t0                     # same ring contents, restored t_b
    q_all = workloads.normal((steps * B, H, d), 303, 1.0, dt).cuda()
    k_all = workloads.normal((steps * B, Hkv, d), 304, 1.0, dt).cuda()
    v_all = workloads.normal((steps * B, Hkv, d), 305, 1.0, dt).cuda()
    o = torch.empty(steps, B, H, d, dtype=dt, device="cuda")
    lse = torch.empty(steps, B, H, device="cuda")
    for s in range(steps):                   # enqueued back to back
        q, k, v = (x[s * B:(s + 1) * B] for x in (q_all, k_all, v_all))
        if fused:
            cache.decode_step_fused(q, k, v, o[s], lse[s])
        else:
            cache.append_kv(k, v)
            cache.decode_step(q, o[s], lse[s])
    torch.cuda.synchronize()
    assert cache.sync_status() == 0
    for s in range(steps):
        for b in range(B):
            sl = s * B + b
            states[b], ro, rl = oracle.decode_step_fused(
                states[b], f64(q_all[sl]), f64(k_all[sl]), f64(v_all[sl]), n)
            assert_close(f64(o[s, b]), ro, dtype, f"step {s} seq {b}")
            assert np.abs(f64(lse[s, b]) - rl).max() <= (1e-4 if dtype == 0 else 1e-3)
    t_end = (t0 or 0) + steps
    for b, m in enumerate(m_list):
        assert cache.get_t(b) == t_end
        assert cache.cache_len(b) == oracle.cache_len(m, n, t_end)
    # the ring holds exactly the oracle's slots
    Ks, Vs = cache.slabs()
    m_cap = max(m_list)
    for b in range(B):
        held = sorted(oracle.ring_outputs(t_end, n))
        np.testing.assert_array_equal(
            f64(Ks[b, :, m_cap:])[:, held].transpose(1, 0, 2), states[b]["Kr"][held])
        np.testing.assert_array_equal(
            f64(Vs[b, :, m_cap:])[:, held].transpose(1, 0, 2), states[b]["Vr"][held])


def test_stream_decode_after_reprefill(cuda_lib):
    """The first decode launch after a prefill may not read the prefix before
    its dependency wait; later ones may.  Prefill prefix A, decode, prefill a
    different prefix B into the same long cache and decode at once, all
    back to back on one stream."""
    rswa = cuda_lib
    m, n, H, d, steps = 4128, 128, 8, 128, 3      # 17 MB: the streaming kernel
    cache = rswa.RswaCache(m, n, H, d, 1, rswa.RSWA_BF16)
    outs, refs = [], []
    for seed in (41, 42):
        K = workloads.normal((m, H, d), seed, 1.0, torch.bfloat16)
        V = workloads.normal((m, H, d), seed + 100, 1.0, torch.bfloat16)
        q = workloads.normal((steps, H, d), seed + 200, 1.0, torch.bfloat16)
        k = workloads.normal((steps, H, d), seed + 300, 1.0, torch.bfloat16)
        v = workloads.normal((steps, H, d), seed + 400, 1.0, torch.bfloat16)
        cache.prefill(None, K.cuda(), V.cuda(), None, [m], 0)
        o = torch.empty(steps, 1, H, d, dtype=torch.bfloat16, device="cuda")
        for s in range(steps):
            cache.decode_step_fused(q[s][None].cuda(), k[s][None].cuda(),
                                    v[s][None].cuda(), o[s])
        outs.append(o)
        st = oracle.prefill_cache(f64(K), f64(V), m, n, 0)
        r = []
        for s in range(steps):
            st, ro, _ = oracle.decode_step_fused(st, f64(q[s]), f64(k[s]), f64(v[s]), n)
            r.append(ro)
        refs.append(np.stack(r))
    torch.cuda.synchronize()
    assert cache.sync_status() == 0
    for o, r in zip(outs, refs):
        assert_close(f64(o[:, 0]), r, 1, "after prefill")


def test_gqa_tc_back_to_back(cuda_lib):
    """Several fused grouped-head steps on the tensor cores enqueued back to
    back at a batched shape (more CTAs than one wave, two per SM sharing its
    TMEM): each step's next-launch trigger fires right after its dependency
    wait.  Every step is checked against the oracle."""
    rswa = cuda_lib
    B, H, Hkv, d, n, steps = 48, 16, 4, 128, 128, 4
    m_list = workloads.prefix_lengths(B, 200, 1400, seed=11)
    T = 130                                  # the ring has wrapped once
    rows = [m + T for m in m_list]
    K = workloads.normal((sum(rows), Hkv, d), 311, 1.0, torch.bfloat16)
    V = workloads.normal((sum(rows), Hkv, d), 312, 1.0, torch.bfloat16)
    cache = rswa.RswaCache(max(m_list), n, H, d, B, rswa.RSWA_BF16, kv_heads=Hkv)
    cache.prefill(None, K.cuda(), V.cuda(), None, m_list, T)
    offs = np.cumsum([0] + rows)
    states = [oracle.prefill_cache(f64(K[offs[b]:offs[b + 1]]),
                                   f64(V[offs[b]:offs[b + 1]]), m_list[b], n, T)
              for b in range(B)]
    q_all = workloads.normal((steps * B, H, d), 313, 1.0, torch.bfloat16).cuda()
    k_all = workloads.normal((steps * B, Hkv, d), 314, 1.0, torch.bfloat16).cuda()
    v_all = workloads.normal((steps * B, Hkv, d), 315, 1.0, torch.bfloat16).cuda()
    o = torch.empty(steps, B, H, d, dtype=torch.bfloat16, device="cuda")
    for s in range(steps):
        cache.decode_step_fused(*(x[s * B:(s + 1) * B] for x in (q_all, k_all, v_all)),
                                o[s])
    torch.cuda.synchronize()
    assert cache.sync_status() == 0
    for s in range(steps):
        got = f64(o[s])
        for b in range(B):
            sl = s * B + b
            states[b], ro, _ = oracle.decode_step_fused(
                states[b], f64(q_all[sl]), f64(k_all[sl]), f64(v_all[sl]), n)
            assert_close(got[b], ro, 1, f"step {s} seq {b}")
    for b in range(B):
        assert cache.get_t(b) == T + steps


# ---------------------------------------------------------------------------
# blocks of consecutive outputs, also longer than the window (chunked prefill
# of output text into an existing cache)
# ---------------------------------------------------------------------------

CHUNK_CASES = [
    # (m_list, n, H, Hkv, d, dtype, t0, blocks)  t0 outputs decoded first
    ([288], 128, 10, 10, 128, 1, 0, [129]),                  # n + 1, empty ring
    ([288], 128, 10, 10, 128, 1, 37, [391, 16]),             # 3n + 7, then 16
    ([1056], 128, 4, 4, 128, 1, 200, [1000]),                # the ring wrapped
    ([0], 128, 4, 4, 128, 1, 5, [1000, 129]),                # vanilla SWA
    ([288, 0, 1056], 128, 4, 2, 128, 1, 130, [300]),         # ragged, grouped
    ([300], 64, 3, 3, 128, 1, 20, [63, 64, 65]),             # around the TC threshold
    ([0], 128, 4, 4, 128, 1, 0, [64, 100]),                  # split units: 1, then 2 key tiles
    ([1056], 128, 4, 2, 128, 1, 200, [300]),                 # split last unit, wrapped ring, grouped
    ([0, 17, 128, 129, 200, 255, 256, 300], 128, 10, 5, 128, 1, 40, [300]),  # paired tiles: 160 units fill the SMs
    ([100], 7, 2, 2, 64, 1, 3, [20, 9]),                     # d 64: CUDA cores
    ([50], 16, 2, 2, 128, 0, 9, [40]),                       # float32: CUDA cores
]


@pytest.mark.parametrize("case", CHUNK_CASES,
                         ids=lambda c: f"m{c[0]}n{c[1]}H{c[2]}kv{c[3]}d{c[4]}t{c[6]}b{c[7]}")
def test_decode_block_any_length(cuda_lib, case):
    """A block of C outputs through rswa_decode_block equals rows
    m + t0 .. m + t0 + C - 1 of the oracle's prefill of the whole sequence;
    afterwards the ring holds the oracle's last n outputs bit-exactly and t_b
    has advanced by C."""
    rswa = cuda_lib
    m_list, n, H, Hkv, d, dtype, t0, blocks = case
    B = len(m_list)
    dt = tdt(dtype)
    T = t0 + sum(blocks)
    rows = [m + T for m in m_list]
    Q = workloads.normal((sum(rows), H, d), 401, 1.0, dt)
    K = workloads.normal((sum(rows), Hkv, d), 402, 1.0, dt)
    V = workloads.normal((sum(rows), Hkv, d), 403, 1.0, dt)
    offs = np.cumsum([0] + rows)
    seq = [slice(offs[b], offs[b + 1]) for b in range(B)]
    cache = rswa.RswaCache(max(m_list), n, H, d, B, dtype, kv_heads=Hkv)
    # the prefix and the first t0 outputs by prefill
    pk = torch.cat([K[s][:m + t0] for s, m in zip(seq, m_list)]).cuda()
    pv = torch.cat([V[s][:m + t0] for s, m in zip(seq, m_list)]).cuda()
    cache.prefill(None, pk, pv, None, m_list, t0)
    refs = [oracle.prefill_attention(f64(Q[s]), f64(K[s]), f64(V[s]), m, n)
            for s, m in zip(seq, m_list)]
    t = t0
    for C in blocks:
        q, k, v = (torch.stack([x[s][m + t:m + t + C] for s, m in zip(seq, m_list)])
                   .contiguous().cuda() for x in (Q, K, V))
        o = torch.empty_like(q)
        lse = torch.empty(B, C, H, device="cuda")
        cache.decode_block(q, k, v, o, lse)
        torch.cuda.synchronize()
        for b, m in enumerate(m_list):
            assert_close(f64(o[b]), refs[b][0][m + t:m + t + C], dtype,
                         f"block at t={t} seq {b}")
            assert np.abs(f64(lse[b]) - refs[b][1][m + t:m + t + C]).max() <= \
                (1e-4 if dtype == 0 else 1e-3)
        t += C
        for b in range(B):
            assert cache.get_t(b) == t
    assert cache.sync_status() == 0
    Ks, Vs = cache.slabs()
    m_cap = max(m_list)
    for b, (s, m) in enumerate(zip(seq, m_list)):
        st = oracle.prefill_cache(f64(K[s]), f64(V[s]), m, n, T)
        held = sorted(oracle.ring_outputs(T, n))
        np.testing.assert_array_equal(
            f64(Ks[b, :, m_cap:])[:, held].transpose(1, 0, 2), st["Kr"][held])
        np.testing.assert_array_equal(
            f64(Vs[b, :, m_cap:])[:, held].transpose(1, 0, 2), st["Vr"][held])
        np.testing.assert_array_equal(f64(Ks[b, :, :m]).transpose(1, 0, 2), st["Kp"])
        assert cache.cache_len(b) == oracle.cache_len(m, n, T)


GQA_TC_CASES = [
    # (B, H, Hkv, m_lo, m_hi, n, T0): the tensor-core grouped decode's forms
    (24, 32, 8, 100, 1500, 128, 130),     # stream-K: ragged heads split over CTAs
    (3, 8, 2, 0, 40, 1024, 5),            # stream-K: tiny, most CTAs without work
    (300, 8, 2, 50, 400, 64, 70),         # B > 256: one CTA per chunk
    (24, 32, 2, 200, 900, 128, 20),       # 16 heads per KV head: one CTA per chunk
    (16, 24, 8, 700, 2100, 256, 300),     # 3 heads per KV head, two-tile wrapped ring
    (12, 16, 8, 300, 1500, 128, 140),     # stream-K, 2 heads per KV head (G = 2)
    (10, 48, 6, 300, 1500, 128, 140),     # stream-K, 8 heads per KV head (G = 8)
    (260, 4, 2, 20, 300, 64, 70),         # B > 256, one CTA per chunk, G = 2
    (260, 16, 2, 20, 300, 64, 70),        # B > 256, one CTA per chunk, G = 8
]


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("case", GQA_TC_CASES, ids=lambda c: f"B{c[0]}H{c[1]}kv{c[2]}n{c[5]}")
def test_gqa_tc_forms(cuda_lib, case, fused):
    """The grouped tensor-core decode in its stream-K form (persistent CTAs
    over the key tiles of all KV heads) and its one-CTA-per-chunk form,
    against the oracle over a few back-to-back steps."""
    rswa = cuda_lib
    B, H, Hkv, m_lo, m_hi, n, T0 = case
    d, steps = 128, 3
    m_list = workloads.prefix_lengths(B, m_lo, m_hi, seed=B + H)
    rows = [m + T0 for m in m_list]
    K = workloads.normal((sum(rows), Hkv, d), 321, 1.0, torch.bfloat16)
    V = workloads.normal((sum(rows), Hkv, d), 322, 1.0, torch.bfloat16)
    cache = rswa.RswaCache(max(m_list), n, H, d, B, rswa.RSWA_BF16, kv_heads=Hkv)
    cache.prefill(None, K.cuda(), V.cuda(), None, m_list, T0)
    offs = np.cumsum([0] + rows)
    states = [oracle.prefill_cache(f64(K[offs[b]:offs[b + 1]]),
                                   f64(V[offs[b]:offs[b + 1]]), m_list[b], n, T0)
              for b in range(B)]
    q_all = workloads.normal((steps * B, H, d), 323, 1.0, torch.bfloat16).cuda()
    k_all = workloads.normal((steps * B, Hkv, d), 324, 1.0, torch.bfloat16).cuda()
    v_all = workloads.normal((steps * B, Hkv, d), 325, 1.0, torch.bfloat16).cuda()
    o = torch.empty(steps, B, H, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(steps, B, H, device="cuda")
    for s in range(steps):
        q, k, v = (x[s * B:(s + 1) * B] for x in (q_all, k_all, v_all))
        if fused:
            cache.decode_step_fused(q, k, v, o[s], lse[s])
        else:
            cache.append_kv(k, v)
            cache.decode_step(q, o[s], lse[s])
    torch.cuda.synchronize()
    assert cache.sync_status() == 0
    check = range(B) if B <= 32 else range(0, B, 13)
    for s in range(steps):
        got, gl = f64(o[s]), f64(lse[s])
        for b in range(B):
            sl = s * B + b
            states[b], ro, rl = oracle.decode_step_fused(
                states[b], f64(q_all[sl]), f64(k_all[sl]), f64(v_all[sl]), n)
            if b in check:
                assert_close(got[b], ro, 1, f"step {s} seq {b}")
                assert np.abs(gl[b] - rl).max() <= 1e-3
    for b in range(B):
        assert cache.get_t(b) == T0 + steps
