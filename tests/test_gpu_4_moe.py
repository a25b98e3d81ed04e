"""GPU parity of the whole MoE forward (moe_forward through the C ABI) against
the oracle, on the workloads' MoE shapes (including the DeepSeek-V4 routed-expert
shape).

tiny: every token; decode/prefill/skewed: the routing, the permutation and the
quantized activations of every token are compared bit for bit, and the output
rows of a seeded sample of tokens against the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import (assert_close_tol, cosine, padded_rows_of_compact, sf_rows_index)
from nvfp4_block_scaled_05_gb300 import binding as B
from nvfp4_block_scaled_05_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _ws_view(ws, lay, name, dtype, count):
    off = lay[name]
    itemsize = torch.empty((), dtype=dtype).element_size()
    return ws[off:off + count * itemsize].view(dtype)


def _run(cfg, seed, sample):
    inp = W.moe_inputs(cfg, seed=seed, device=DEV)
    wts = B.prepare_moe_weights(inp["w1"], inp["w2"])
    gs_h = torch.tensor([cfg.gs_h], dtype=torch.float32, device=DEV)
    T, K, I, E, k = cfg.T, cfg.K, cfg.I, cfg.E, cfg.k
    ws = torch.empty(B.moe_forward_workspace_size(T, K, I, E, k), dtype=torch.uint8, device=DEV)
    y = B.moe_forward(inp["x"], inp["logits"], wts, k, gs_h, ws=ws)
    assert B.nvfp4moe_last_device_status() == 0
    lay = B.moe_forward_workspace_layout(T, K, I, E, k)
    x = W.bf16_bits(inp["x"])
    logits = inp["logits"].cpu().numpy()
    w1_dev, w2_dev = inp["w1"], inp["w2"]
    tokens = (np.arange(T) if sample is None else
              np.sort(np.random.default_rng(seed + 99).choice(T, sample, replace=False)))
    ref = O.moe_forward(x, logits, lambda e: W.bf16_bits(w1_dev[e]), lambda e: W.bf16_bits(w2_dev[e]),
                        k, np.float32(cfg.gs_h), tokens=tokens)
    M = T * k
    # bit-exact intermediates
    assert np.array_equal(_ws_view(ws, lay, "topk_ids", torch.int32, M).cpu().numpy().reshape(T, k), ref["ids"])
    tw = _ws_view(ws, lay, "topk_w", torch.float32, M).cpu().numpy().reshape(T, k)
    assert np.allclose(tw, ref["w"], rtol=1e-6, atol=1e-7)
    offsets = _ws_view(ws, lay, "offsets", torch.int32, E + 1).cpu().numpy()
    assert np.array_equal(offsets, ref["offsets"])
    assert np.array_equal(_ws_view(ws, lay, "perm_to_flat", torch.int32, M).cpu().numpy(), ref["perm_to_flat"])
    assert np.array_equal(_ws_view(ws, lay, "flat_to_perm", torch.int32, M).cpu().numpy(), ref["flat_to_perm"])
    assert _ws_view(ws, lay, "gs_x", torch.float32, 1).item() == ref["gs_x"]
    a_rows = lay["a_rows"]
    a_codes = _ws_view(ws, lay, "a_codes", torch.uint8, a_rows * K // 2).view(a_rows, K // 2)
    a_sf = _ws_view(ws, lay, "a_sf", torch.uint8, B.nvfp4_sf_bytes(a_rows, K, B.NVFP4_SF_TILED_ROWS)).cpu().numpy()
    prow = padded_rows_of_compact(offsets)
    # every routed copy of the sampled tokens carries that token's quantized row
    f2p = ref["flat_to_perm"]
    sf_idx = sf_rows_index(a_rows, K)
    for ti, t in enumerate(ref["tokens"]):
        for j in range(k):
            p = prow[f2p[t * k + j]]
            assert np.array_equal(a_codes[p].cpu().numpy(), ref["x_codes"][ti])
            assert np.array_equal(a_sf[sf_idx[p]], ref["x_sf"][ti])
    got = y[torch.from_numpy(np.asarray(ref["tokens"])).to(DEV)].float().cpu().numpy()
    assert_close_tol(got, ref["y"], cfg.name)
    c = cosine(got, ref["y"])
    assert c >= 0.9995, c
    return got, ref, y, inp, wts, gs_h


def test_moe_tiny_every_token():
    got, ref, *_ = _run(W.CONFIGS["tiny"], 0, None)
    # the tolerance above is loose next to tiny outputs; also bound the error
    # by the output's own scale
    rms = np.sqrt(np.mean(ref["y"] ** 2))
    assert np.max(np.abs(got - ref["y"])) <= 0.05 * rms + 2.0 ** -8 * np.abs(ref["y"]).max()


def test_moe_tiny_other_seeds():
    for seed in (1, 2):
        _run(W.CONFIGS["tiny"], seed, None)


def test_moe_decode_sampled():
    _run(W.CONFIGS["decode"], 0, 6)


@pytest.mark.parametrize("name", ["prefill", "skewed"])
def test_moe_prefill_shapes_sampled(name):
    _run(W.CONFIGS[name], 0, 3)


@pytest.mark.parametrize("name,sample", [("dsv4_decode", 4), ("dsv4_prefill", 2)])
def test_moe_deepseek_v4_shape_sampled(name, sample):
    """384 experts, top-6, I=3072: the routed-expert shape of the model the
    pages deploy (gate/up N = 6144, down-projection K = 3072)."""
    _run(W.CONFIGS[name], 0, sample)


def test_moe_edge_shapes():
    """T=1; every token on one expert; more experts than routed rows."""
    for (T, K, I, E, k, mode) in [(1, 256, 64, 8, 2, "rand"), (200, 256, 128, 4, 1, "one"),
                                  (3, 384, 192, 64, 4, "rand")]:
        cfg = W.MoEConfig("edge", T=T, K=K, I=I, E=E, k=k, gs_h=336.0)
        g = torch.Generator(device="cpu").manual_seed(T + E)
        x = torch.randn(T, K, generator=g).to(torch.bfloat16)
        logits = torch.randn(T, E, generator=g)
        if mode == "one":
            logits[:, 2] += 100.0
        w1 = (torch.randn(E, 2 * I, K, generator=g) * 0.05).to(torch.bfloat16)
        w2 = (torch.randn(E, K, I, generator=g) * 0.05).to(torch.bfloat16)
        wts = B.prepare_moe_weights(w1.to(DEV), w2.to(DEV))
        gs_h = torch.tensor([cfg.gs_h], dtype=torch.float32, device=DEV)
        y = B.moe_forward(x.to(DEV), logits.to(DEV), wts, k, gs_h)
        assert B.nvfp4moe_last_device_status() == 0
        xb, w1b, w2b = W.bf16_bits(x), W.bf16_bits(w1), W.bf16_bits(w2)
        ref = O.moe_forward(xb, logits.numpy(), lambda e: w1b[e], lambda e: w2b[e], k, np.float32(cfg.gs_h))
        got = y.float().cpu().numpy()
        assert_close_tol(got, ref["y"], "edge %s" % ((T, E, k, mode),))
        assert cosine(got, ref["y"]) >= 0.9995


def test_moe_random_shapes_sweep():
    """Seeded random shapes through the whole forward (T from 1 to ~700, K and I
    multiples of 128 and 64 with ragged 512-element chunks, E from k to 64, k
    from 1 to 8), every token against the oracle; each shape also with the 2-SM
    pair GEMMs (used where the weight tiles are whole 256-row tiles), which
    must give the same bits as the default kernel."""
    rng = np.random.default_rng(2024)
    for case in range(6):
        k = int(rng.integers(1, 9))
        E = int(rng.integers(max(k, 2), 65))
        tier = case % 3
        T = 1 if tier == 0 else int(rng.integers(2, 64)) if tier == 1 else int(rng.integers(64, 700))
        K = int(rng.choice([128, 256, 384, 640, 1024]))
        I = int(rng.choice([64, 128, 192, 320]))
        cfg = W.MoEConfig("sweep", T=T, K=K, I=I, E=E, k=k, gs_h=336.0)
        g = torch.Generator(device="cpu").manual_seed(1000 + case)
        x = torch.randn(T, K, generator=g).to(torch.bfloat16)
        logits = torch.randn(T, E, generator=g)
        w1 = (torch.randn(E, 2 * I, K, generator=g) * 0.05).to(torch.bfloat16)
        w2 = (torch.randn(E, K, I, generator=g) * 0.05).to(torch.bfloat16)
        wts = B.prepare_moe_weights(w1.to(DEV), w2.to(DEV))
        gs_h = torch.tensor([cfg.gs_h], dtype=torch.float32, device=DEV)
        y = B.moe_forward(x.to(DEV), logits.to(DEV), wts, k, gs_h)
        assert B.nvfp4moe_last_device_status() == 0
        try:
            B.nvfp4moe_set_gemm_mode(1)
            y_pair = B.moe_forward(x.to(DEV), logits.to(DEV), wts, k, gs_h)
        finally:
            B.nvfp4moe_set_gemm_mode(0)
        assert B.nvfp4moe_last_device_status() == 0
        assert torch.equal(y, y_pair), (T, K, I, E, k)
        xb, w1b, w2b = W.bf16_bits(x), W.bf16_bits(w1), W.bf16_bits(w2)
        ref = O.moe_forward(xb, logits.numpy(), lambda e: w1b[e], lambda e: w2b[e], k, np.float32(cfg.gs_h))
        got = y.float().cpu().numpy()
        assert_close_tol(got, ref["y"], "sweep %s" % ((T, K, I, E, k),))
        assert cosine(got, ref["y"]) >= 0.9995, (T, K, I, E, k)


def test_moe_deterministic_and_graph_capturable():
    cfg = W.CONFIGS["tiny"]
    inp = W.moe_inputs(cfg, seed=3, device=DEV)
    wts = B.prepare_moe_weights(inp["w1"], inp["w2"])
    gs_h = torch.tensor([cfg.gs_h], dtype=torch.float32, device=DEV)
    ws = torch.empty(B.moe_forward_workspace_size(cfg.T, cfg.K, cfg.I, cfg.E, cfg.k),
                     dtype=torch.uint8, device=DEV)
    y1 = B.moe_forward(inp["x"], inp["logits"], wts, cfg.k, gs_h, ws=ws).clone()
    y2 = B.moe_forward(inp["x"], inp["logits"], wts, cfg.k, gs_h, ws=ws).clone()
    assert torch.equal(y1, y2)
    y3 = torch.empty_like(y1)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        B.moe_forward(inp["x"], inp["logits"], wts, cfg.k, gs_h, ws=ws, y=y3)  # warm-up on the stream
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            B.moe_forward(inp["x"], inp["logits"], wts, cfg.k, gs_h, ws=ws, y=y3)
    torch.cuda.current_stream().wait_stream(s)
    y3.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y1, y3)
    assert B.nvfp4moe_last_device_status() == 0


def test_moe_largest_expert_count_and_topk():
    """E=1024 experts with top-16 (the largest the entry points accept) and
    E=1024 with top-1, against the oracle for every token."""
    for (T, K, I, E, k) in [(8, 256, 64, 1024, 16), (40, 128, 64, 1024, 1)]:
        cfg = W.MoEConfig("max", T=T, K=K, I=I, E=E, k=k, gs_h=336.0)
        g = torch.Generator(device="cpu").manual_seed(E + k)
        x = torch.randn(T, K, generator=g).to(torch.bfloat16)
        logits = torch.randn(T, E, generator=g)
        w1 = (torch.randn(E, 2 * I, K, generator=g) * 0.05).to(torch.bfloat16)
        w2 = (torch.randn(E, K, I, generator=g) * 0.05).to(torch.bfloat16)
        wts = B.prepare_moe_weights(w1.to(DEV), w2.to(DEV))
        gs_h = torch.tensor([cfg.gs_h], dtype=torch.float32, device=DEV)
        y = B.moe_forward(x.to(DEV), logits.to(DEV), wts, k, gs_h)
        assert B.nvfp4moe_last_device_status() == 0
        xb, w1b, w2b = W.bf16_bits(x), W.bf16_bits(w1), W.bf16_bits(w2)
        ref = O.moe_forward(xb, logits.numpy(), lambda e: w1b[e], lambda e: w2b[e], k, np.float32(cfg.gs_h))
        got = y.float().cpu().numpy()
        assert_close_tol(got, ref["y"], "E=%d k=%d" % (E, k))
        assert cosine(got, ref["y"]) >= 0.9995


def test_fused_dispatch_choice():
    """moe_forward takes the fused dispatch whenever its cooperative kernel's
    co-resident blocks hold the tokens (above FRONT_FUSED_QUANTIZE_MAX_ROWS
    routed rows its quantize + scatter is a second kernel), and the separate
    kernels beyond that."""
    for T in (1, 128, 8192, 16384):
        assert B.moe_forward_uses_fused_dispatch(T, 256, 8)
        assert B.moe_dispatch_supported(T, 256, 8)
    # 1.6M routed rows: more than 4096 slots per co-resident block
    assert not B.moe_dispatch_supported(200000, 256, 8)
    assert not B.moe_forward_uses_fused_dispatch(200000, 256, 8)


def test_moe_skewed_heaviest_expert_every_tile():
    """The full-size skewed prefill (T=16384, Zipf(1.2) popularity, 16 experts
    never chosen): the L2 output rows of the heaviest expert (~15k routed rows,
    ~117 activation tiles of 128) element by element against the fp64 oracle,
    16 rows in EVERY one of its activation tiles (each tile's first and last
    row and 14 seeded others, the ragged last tile included), and every routed
    row of the three lightest active experts (single-tile groups). The oracle
    runs only the sampled rows (about 2000 of the 131072), so the case stays
    within seconds; all columns are compared."""
    cfg = W.CONFIGS["skewed"]
    inp = W.moe_inputs(cfg, seed=0, device=DEV)
    wts = B.prepare_moe_weights(inp["w1"], inp["w2"])
    gs_h = torch.tensor([cfg.gs_h], dtype=torch.float32, device=DEV)
    T, K, I, E, k = cfg.T, cfg.K, cfg.I, cfg.E, cfg.k
    ws = torch.empty(B.moe_forward_workspace_size(T, K, I, E, k), dtype=torch.uint8, device=DEV)
    B.moe_forward(inp["x"], inp["logits"], wts, k, gs_h, ws=ws)
    assert B.nvfp4moe_last_device_status() == 0
    lay = B.moe_forward_workspace_layout(T, K, I, E, k)
    M = T * k
    offsets = _ws_view(ws, lay, "offsets", torch.int32, E + 1).cpu().numpy()
    p2f = _ws_view(ws, lay, "perm_to_flat", torch.int32, M).cpu().numpy()
    f2p = _ws_view(ws, lay, "flat_to_perm", torch.int32, M).cpu().numpy()
    counts = np.diff(offsets)
    heavy = int(np.argmax(counts))
    light = [int(e) for e in np.argsort(counts, kind="stable") if counts[e] > 0][:3]
    assert counts[heavy] > 4096 and all(counts[e] <= 128 for e in light)
    rng = np.random.default_rng(17)
    rows = []
    n = int(counts[heavy])
    for t0 in range(0, n, 128):
        t1 = min(n, t0 + 128)
        pick = {t0, t1 - 1} | set(rng.choice(np.arange(t0, t1), min(14, t1 - t0), replace=False).tolist())
        rows += [int(offsets[heavy]) + r for r in sorted(pick)]
    for e in light:
        rows += list(range(int(offsets[e]), int(offsets[e + 1])))
    tokens = sorted(set(int(p2f[r]) // k for r in rows))
    x = W.bf16_bits(inp["x"])
    w1_dev, w2_dev = inp["w1"], inp["w2"]
    ref = O.moe_forward(x, inp["logits"].cpu().numpy(), lambda e: W.bf16_bits(w1_dev[e]),
                        lambda e: W.bf16_bits(w2_dev[e]), k, np.float32(cfg.gs_h), tokens=tokens,
                        experts={heavy, *light}, keep=True)
    assert np.array_equal(ref["offsets"], offsets)
    out = _ws_view(ws, lay, "out", torch.bfloat16, M * K).view(M, K)
    want_rows = set(rows)
    idx, want = [], []
    for (t, j), d in ref["inter"].items():
        r = int(f2p[t * k + j])
        if r in want_rows:
            idx.append(r)
            want.append(d["o"])
    assert len(idx) == len(want_rows)
    got = out[torch.tensor(idx, device=DEV)].float().cpu().numpy()
    want = np.array(want)
    assert_close_tol(got, want, "skewed heaviest expert %d and experts %s" % (heavy, light))
    assert cosine(got, want) >= 0.9995
