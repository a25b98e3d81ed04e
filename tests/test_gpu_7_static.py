"""GPU parity of moe_forward_static: the forward with a pre-computed activation
global scale, whose route + permute + quantize + scatter run as one
cooperative kernel.

* With gs_x equal to the one moe_forward computes, every intermediate (routing,
  permutation, offsets, the quantized rows) and y are bit-identical to
  moe_forward's.
* With another gs_x, the intermediates equal the oracle's (given that gs_x) bit
  for bit and y is within the tolerance.
* Captured in a CUDA graph and replayed on new inputs, it gives the eager
  result bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import assert_close_tol, cosine, padded_rows_of_compact, sf_rows_index
from nvfp4_block_scaled_05_gb300 import binding as B
from nvfp4_block_scaled_05_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
NAMES = ["topk_ids", "topk_w", "offsets", "perm_to_flat", "flat_to_perm"]


def _view(ws, lay, name, dtype, count):
    off = lay[name]
    n = torch.empty((), dtype=dtype).element_size()
    return ws[off:off + count * n].view(dtype)


def _inter(ws, lay, T, K, E, k):
    M = T * k
    d = {n: _view(ws, lay, n, torch.int32 if n != "topk_w" else torch.float32, E + 1 if n == "offsets" else M)
         .cpu().numpy().copy() for n in NAMES}
    a_rows = lay["a_rows"]
    prow = padded_rows_of_compact(d["offsets"])
    codes = _view(ws, lay, "a_codes", torch.uint8, a_rows * K // 2).view(a_rows, K // 2).cpu().numpy()
    sf = _view(ws, lay, "a_sf", torch.uint8, B.nvfp4_sf_bytes(a_rows, K, B.NVFP4_SF_TILED_ROWS)).cpu().numpy()
    d["rows"] = codes[prow]
    d["sf"] = sf[sf_rows_index(a_rows, K)][prow]
    return d


def _setup(cfg, seed=0):
    inp = W.moe_inputs(cfg, seed=seed, device=DEV)
    wts = B.prepare_moe_weights(inp["w1"], inp["w2"])
    gs_h = torch.tensor([cfg.gs_h], dtype=torch.float32, device=DEV)
    nb = B.moe_forward_workspace_size(cfg.T, cfg.K, cfg.I, cfg.E, cfg.k)
    lay = B.moe_forward_workspace_layout(cfg.T, cfg.K, cfg.I, cfg.E, cfg.k)
    return inp, wts, gs_h, nb, lay


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "dsv4_decode"])
def test_static_equals_dynamic_with_same_gs(name):
    cfg = W.CONFIGS[name]
    inp, wts, gs_h, nb, lay = _setup(cfg)
    ws1 = torch.empty(nb, dtype=torch.uint8, device=DEV)
    ws2 = torch.full((nb,), 0xAB, dtype=torch.uint8, device=DEV)   # stale bytes
    y1 = B.moe_forward(inp["x"], inp["logits"], wts, cfg.k, gs_h, ws=ws1)
    gs_x = _view(ws1, lay, "gs_x", torch.float32, 1).clone()
    y2 = B.moe_forward_static(inp["x"], inp["logits"], wts, cfg.k, gs_h, gs_x, ws=ws2)
    assert B.nvfp4moe_last_device_status() == 0
    a = _inter(ws1, lay, cfg.T, cfg.K, cfg.E, cfg.k)
    b = _inter(ws2, lay, cfg.T, cfg.K, cfg.E, cfg.k)
    for n in a:
        assert np.array_equal(a[n], b[n]), n
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("name,sample", [("tiny", None), ("decode", 4)])
def test_static_matches_oracle_with_given_gs(name, sample):
    cfg = W.CONFIGS[name]
    inp, wts, gs_h, nb, lay = _setup(cfg, seed=1)
    xb = W.bf16_bits(inp["x"])
    g = np.float32(O.global_scale(O.amax_bf16(xb)) * np.float32(0.75))   # not the computed one
    ws = torch.empty(nb, dtype=torch.uint8, device=DEV)
    y = B.moe_forward_static(inp["x"], inp["logits"], wts, cfg.k, gs_h,
                             torch.tensor([g], dtype=torch.float32, device=DEV), ws=ws)
    assert B.nvfp4moe_last_device_status() == 0
    T, k = cfg.T, cfg.k
    tokens = (np.arange(T) if sample is None else
              np.sort(np.random.default_rng(7).choice(T, sample, replace=False)))
    w1, w2 = inp["w1"], inp["w2"]
    ref = O.moe_forward(xb, inp["logits"].cpu().numpy(), lambda e: W.bf16_bits(w1[e]),
                        lambda e: W.bf16_bits(w2[e]), k, np.float32(cfg.gs_h), tokens=tokens, gs_x=g)
    d = _inter(ws, lay, T, cfg.K, cfg.E, k)
    assert np.array_equal(d["topk_ids"].reshape(T, k), ref["ids"])
    assert np.allclose(d["topk_w"].reshape(T, k), ref["w"], rtol=1e-6, atol=1e-7)
    assert np.array_equal(d["offsets"], ref["offsets"])
    assert np.array_equal(d["perm_to_flat"], ref["perm_to_flat"])
    assert np.array_equal(d["flat_to_perm"], ref["flat_to_perm"])
    f2p = ref["flat_to_perm"]
    for ti, t in enumerate(ref["tokens"]):
        for j in range(k):
            assert np.array_equal(d["rows"][f2p[t * k + j]], ref["x_codes"][ti])
            assert np.array_equal(d["sf"][f2p[t * k + j]], ref["x_sf"][ti])
    got = y[torch.from_numpy(np.asarray(ref["tokens"])).to(DEV)].float().cpu().numpy()
    assert_close_tol(got, ref["y"], name)
    assert cosine(got, ref["y"]) >= 0.9995


def test_static_edge_shapes():
    """T=1 (one block), all tokens on one expert, E above the routed rows, and
    E=1000 (32 logits per lane)."""
    for (T, K, I, E, k, mode) in [(1, 256, 64, 8, 2, "rand"), (200, 256, 128, 4, 1, "one"),
                                  (3, 384, 192, 64, 4, "rand"), (700, 128, 64, 1000, 3, "rand")]:
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
        nb = B.moe_forward_workspace_size(T, K, I, E, k)
        ws1 = torch.empty(nb, dtype=torch.uint8, device=DEV)
        y1 = B.moe_forward(x.to(DEV), logits.to(DEV), wts, k, gs_h, ws=ws1)
        lay = B.moe_forward_workspace_layout(T, K, I, E, k)
        gs_x = _view(ws1, lay, "gs_x", torch.float32, 1).clone()
        ws2 = torch.empty(nb, dtype=torch.uint8, device=DEV)
        y2 = B.moe_forward_static(x.to(DEV), logits.to(DEV), wts, k, gs_h, gs_x, ws=ws2)
        assert B.nvfp4moe_last_device_status() == 0
        a, b = _inter(ws1, lay, T, K, E, k), _inter(ws2, lay, T, K, E, k)
        for n in a:
            assert np.array_equal(a[n], b[n]), (n, T, E, k)
        assert torch.equal(y1, y2), (T, E, k)


@pytest.mark.parametrize("name", ["decode", "front_two_kernels"])
def test_static_graph_replay_on_new_inputs(name):
    """moe_forward_static captured in a CUDA graph and replayed on new inputs
    copied into the captured buffers equals the eager call bit for bit.
    "front_two_kernels" has more routed rows than FRONT_FUSED_QUANTIZE_MAX_ROWS,
    so the captured front is the cooperative kernel plus the quantize kernel."""
    if name == "decode":
        cfg = W.CONFIGS["decode"]
    else:
        T = B.FRONT_FUSED_QUANTIZE_MAX_ROWS // 8 + 40
        cfg = W.MoEConfig(name, T=T, K=256, I=128, E=16, k=8, gs_h=1344.0)
    inp, wts, gs_h, nb, lay = _setup(cfg, seed=2)
    inp2 = W.moe_inputs(cfg, seed=3, device=DEV, weights=False)
    gs_x = torch.tensor([2688.0 / 4.5], dtype=torch.float32, device=DEV)
    ws = torch.empty(nb, dtype=torch.uint8, device=DEV)
    x_s, l_s = inp["x"].clone(), inp["logits"].clone()
    y_s = torch.empty_like(inp["x"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        B.moe_forward_static(x_s, l_s, wts, cfg.k, gs_h, gs_x, ws=ws, y=y_s)   # warm-up
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            B.moe_forward_static(x_s, l_s, wts, cfg.k, gs_h, gs_x, ws=ws, y=y_s)
    torch.cuda.current_stream().wait_stream(s)
    for src in (inp, inp2):
        x_s.copy_(src["x"])
        l_s.copy_(src["logits"])
        graph.replay()
        torch.cuda.synchronize()
        eager = B.moe_forward_static(src["x"], src["logits"], wts, cfg.k, gs_h, gs_x)
        assert B.nvfp4moe_last_device_status() == 0
        assert torch.equal(y_s, eager)


def test_dynamic_graph_replay_two_kernel_front():
    """moe_forward (the global scale of x computed every call) captured in a
    CUDA graph at more routed rows than FRONT_FUSED_QUANTIZE_MAX_ROWS (the
    front's counter reset, cooperative kernel and quantize kernel are all
    graph nodes), replayed on new inputs: bit for bit the eager result."""
    T = B.FRONT_FUSED_QUANTIZE_MAX_ROWS // 8 + 40
    cfg = W.MoEConfig("front_two_kernels", T=T, K=256, I=128, E=16, k=8, gs_h=1344.0)
    assert B.moe_forward_uses_fused_dispatch(cfg.T, cfg.E, cfg.k)
    inp, wts, gs_h, nb, lay = _setup(cfg, seed=6)
    inp2 = W.moe_inputs(cfg, seed=7, device=DEV, weights=False)
    ws = torch.empty(nb, dtype=torch.uint8, device=DEV)
    x_s, l_s = inp["x"].clone(), inp["logits"].clone()
    y_s = torch.empty_like(inp["x"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        B.moe_forward(x_s, l_s, wts, cfg.k, gs_h, ws=ws, y=y_s)   # warm-up
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            B.moe_forward(x_s, l_s, wts, cfg.k, gs_h, ws=ws, y=y_s)
    torch.cuda.current_stream().wait_stream(s)
    for src in (inp, inp2):
        x_s.copy_(src["x"])
        l_s.copy_(src["logits"])
        graph.replay()
        torch.cuda.synchronize()
        eager = B.moe_forward(src["x"], src["logits"], wts, cfg.k, gs_h)
        assert B.nvfp4moe_last_device_status() == 0
        assert torch.equal(y_s, eager)


def _split_and_fused(cfg, x, logits):
    """Stages 1-2 of the forward twice into two workspaces of moe_forward's
    layout: as the separate route, permute and quantize calls, and as the
    fused dispatch kernel with the global scale computed in it."""
    import ctypes
    T, K, I, E, k = cfg.T, cfg.K, cfg.I, cfg.E, cfg.k
    L = B.lib()
    nb = B.moe_forward_workspace_size(T, K, I, E, k)
    lay = B.moe_forward_workspace_layout(T, K, I, E, k)
    a_rows = lay["a_rows"]
    up = lambda v: -(-v // 256) * 256
    out = []
    for fused in (False, True):
        ws = torch.full((nb,), 0xAB, dtype=torch.uint8, device=DEV)   # stale bytes
        base = ws.data_ptr()
        p = {n: ctypes.c_void_p(base + o) for n, o in lay.items() if n != "a_rows"}
        scratch = base + lay["out"] + up(T * k * K * 2)
        s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        xp, lp = ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(logits.data_ptr())
        if fused:
            st = L.moe_dispatch(xp, K, lp, T, K, E, k, p["gs_x"], p["topk_ids"], p["topk_w"], p["offsets"],
                                p["perm_to_flat"], p["flat_to_perm"], p["a_codes"], p["a_sf"], a_rows,
                                ctypes.c_void_p(scratch), nb - (scratch - base), s)
            assert st == 0, st
        else:
            pb = int(L.moe_permute_workspace_size(T, k, E))
            assert L.moe_route_topk(lp, T, E, k, p["topk_ids"], p["topk_w"], s) == 0
            assert L.moe_permute(p["topk_ids"], T, k, E, p["offsets"], p["perm_to_flat"], p["flat_to_perm"],
                                 ctypes.c_void_p(scratch), pb, s) == 0
            dws = scratch + up(pb)
            assert L.moe_quantize_dispatch(xp, T, K, K, k, E, p["topk_ids"], p["offsets"], p["flat_to_perm"],
                                           None, p["gs_x"], p["a_codes"], p["a_sf"], a_rows,
                                           ctypes.c_void_p(dws), int(L.moe_quantize_dispatch_workspace_size(E)),
                                           s) == 0
        assert B.nvfp4moe_last_device_status() == 0
        d = _inter(ws, lay, T, K, E, k)
        d["gs_x"] = _view(ws, lay, "gs_x", torch.float32, 1).item()
        out.append(d)
    return out


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "skewed", "dsv4_decode"])
def test_fused_dispatch_equals_separate_calls(name):
    """moe_dispatch (the cooperative kernel, the global scale of x computed in
    it; prefill and skewed with the quantize + scatter as a second kernel)
    writes the same bits as moe_route_topk + moe_permute +
    moe_quantize_dispatch: routing, permutation, offsets, gs_x, and every
    routed row's codes and scales."""
    cfg = W.CONFIGS[name]
    assert B.moe_dispatch_supported(cfg.T, cfg.E, cfg.k)
    inp = W.moe_inputs(cfg, seed=5, device=DEV, weights=False)
    split, fused = _split_and_fused(cfg, inp["x"], inp["logits"])
    assert fused["gs_x"] == split["gs_x"]
    for n in NAMES + ["rows", "sf"]:
        assert np.array_equal(fused[n], split[n]), n


def test_fused_dispatch_edge_shapes():
    """T=1; more experts than routed rows (E=1000); every token on one expert;
    an all-zero x (global scale 1); the largest |x| a negative element."""
    for (T, K, E, k, mode) in [(1, 256, 8, 2, "rand"), (3, 384, 1000, 4, "rand"), (200, 256, 4, 1, "one"),
                               (64, 512, 16, 2, "zero"), (96, 256, 8, 2, "negmax")]:
        cfg = W.MoEConfig("edge", T=T, K=K, I=64, E=E, k=k, gs_h=336.0)
        g = torch.Generator(device="cpu").manual_seed(T + E)
        x = torch.randn(T, K, generator=g).to(torch.bfloat16)
        if mode == "zero":
            x.zero_()
        if mode == "negmax":
            x[T // 2, K - 3] = -40.0
        logits = torch.randn(T, E, generator=g)
        if mode == "one":
            logits[:, 2] += 100.0
        split, fused = _split_and_fused(cfg, x.to(DEV), logits.to(DEV))
        assert fused["gs_x"] == split["gs_x"], (T, E)
        if mode == "zero":
            assert fused["gs_x"] == 1.0
        if mode == "negmax":
            assert fused["gs_x"] == O.global_scale(O.amax_bf16(W.bf16_bits(x))) == np.float32(2688.0 / 40.0)
        for n in NAMES + ["rows", "sf"]:
            assert np.array_equal(fused[n], split[n]), (n, T, E)


@pytest.mark.parametrize("extra", [0, 1])
def test_fused_dispatch_at_the_quantize_kernel_threshold(extra):
    """T * k exactly FRONT_FUSED_QUANTIZE_MAX_ROWS (quantize + scatter inside
    the cooperative kernel) and one token more (the second kernel): the same
    bits as the separate calls, with the global scale computed."""
    k = 8
    T = B.FRONT_FUSED_QUANTIZE_MAX_ROWS // k + extra
    cfg = W.MoEConfig("threshold", T=T, K=384, I=64, E=24, k=k, gs_h=336.0)
    g = torch.Generator(device="cpu").manual_seed(T)
    x = torch.randn(T, 384, generator=g).to(torch.bfloat16)
    logits = torch.randn(T, 24, generator=g)
    split, fused = _split_and_fused(cfg, x.to(DEV), logits.to(DEV))
    assert fused["gs_x"] == split["gs_x"]
    for n in NAMES + ["rows", "sf"]:
        assert np.array_equal(fused[n], split[n]), n


def test_fused_dispatch_nan_logits():
    """Reading R16 in the fused dispatch: NaN router logits scattered over a
    decode-shaped batch rank as -inf. Routing equals the oracle's (ids bit for
    bit, weights within 1e-6) and every intermediate equals the separate
    calls' bit for bit."""
    cfg = W.CONFIGS["decode"]
    inp = W.moe_inputs(cfg, seed=9, device="cpu", weights=False)
    logits = inp["logits"].numpy().copy()
    rng = np.random.default_rng(12)
    logits[rng.random(logits.shape) < 0.05] = np.nan
    rows = np.arange(0, logits.shape[0], 4)
    logits[rows, np.argmax(np.nan_to_num(logits[rows], nan=-np.inf), axis=1)] = np.nan
    split, fused = _split_and_fused(cfg, inp["x"].to(DEV), torch.from_numpy(logits).to(DEV))
    rid, rw = O.route_topk(logits, cfg.k)
    assert np.array_equal(fused["topk_ids"].reshape(rid.shape), rid)
    assert np.allclose(fused["topk_w"].reshape(rw.shape), rw, rtol=1e-6, atol=1e-7)
    for n in NAMES + ["rows", "sf"]:
        assert np.array_equal(fused[n], split[n]), n
