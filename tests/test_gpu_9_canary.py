"""Out-of-bounds and input-clobber checks without a sanitizer: every output
and workspace lives inside a larger buffer whose guard bytes (64 KB on each
side) hold a known pattern, and every input is compared with a copy; after
each call the guards and the inputs must be unchanged (canary padding)."""
import numpy as np
import pytest
import torch

from nvfp4_block_scaled_05_gb300 import binding as B
from nvfp4_block_scaled_05_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
G = 64 * 1024
PAT = 0xA5


class Guarded:
    """nbytes of device memory (256-byte aligned) between two guard regions."""

    def __init__(self, nbytes, fill=None):
        n = -(-nbytes // 256) * 256
        self.buf = torch.full((G + n + G,), PAT, dtype=torch.uint8, device=DEV)
        self.n = nbytes
        if fill is not None:
            self.buf[G:G + nbytes] = fill

    def view(self, dtype, shape):
        return self.buf[G:G + self.n].view(dtype).view(shape)

    def bytes(self):
        return self.buf[G:G + self.n]

    def intact(self):
        return bool((self.buf[:G] == PAT).all() and (self.buf[G + self.n:] == PAT).all())


def _check(guards, inputs, before):
    torch.cuda.synchronize()
    assert B.nvfp4moe_last_device_status() == 0
    for name, g in guards.items():
        assert g.intact(), "write outside " + name
    for (name, t), c in zip(inputs.items(), before):
        assert torch.equal(t, c), "input changed: " + name


@pytest.mark.parametrize("front", ["dynamic", "static"])
def test_forward_writes_only_its_outputs(front):
    cfg = W.MoEConfig("canary", T=300, K=1024, I=384, E=24, k=4, gs_h=336.0)
    inp = W.moe_inputs(cfg, seed=8, device=DEV)
    wts = B.prepare_moe_weights(inp["w1"], inp["w2"])
    T, K, I, E, k = cfg.T, cfg.K, cfg.I, cfg.E, cfg.k
    ws = Guarded(B.moe_forward_workspace_size(T, K, I, E, k))
    y = Guarded(T * K * 2)
    gs_h = torch.tensor([cfg.gs_h], device=DEV)
    inputs = {"x": inp["x"], "logits": inp["logits"], "gs_h": gs_h,
              **{n: wts[n] for n in ["w1_codes", "w1_sf", "gs_w1", "w2_codes", "w2_sf", "gs_w2"]}}
    before = [t.clone() for t in inputs.values()]
    if front == "dynamic":
        out = B.moe_forward(inp["x"], inp["logits"], wts, k, gs_h, ws=ws.bytes(), y=y.view(torch.bfloat16, (T, K)))
    else:
        gs_x = torch.tensor([300.0], device=DEV)
        inputs["gs_x"] = gs_x
        before.append(gs_x.clone())
        out = B.moe_forward_static(inp["x"], inp["logits"], wts, k, gs_h, gs_x, ws=ws.bytes(),
                                   y=y.view(torch.bfloat16, (T, K)))
    _check({"workspace": ws, "y": y}, inputs, before)
    assert torch.isfinite(out.float()).all()


def test_quantize_gemm_linear_norm_write_only_their_outputs():
    g = torch.Generator(device="cpu").manual_seed(9)
    M, K, N, E = 333, 512, 384, 3
    x = torch.randn(M, K, generator=g).to(torch.bfloat16).to(DEV)
    x_in = x.clone()
    # quantize (rows not a multiple of 128, tiled scales)
    a_rows = B.nvfp4moe_padded_rows(M, E)
    codes = Guarded(a_rows * K // 2, fill=0)
    sf = Guarded(B.nvfp4_sf_bytes(a_rows, K, B.NVFP4_SF_TILED_ROWS), fill=0)
    gs = Guarded(4)
    B.nvfp4_quantize(x, codes=codes.view(torch.uint8, (a_rows, K // 2))[:M], sf=sf.view(torch.uint8, (-1,)),
                     gs_out=gs.view(torch.float32, (1,)), sf_layout=B.NVFP4_SF_TILED_ROWS)
    _check({"codes": codes, "sf": sf, "gs": gs}, {"x": x}, [x_in])
    # grouped GEMM (groups of 100, 0, 233 rows in the padded layout) and the SwiGLU GEMM
    I = N // 2
    w1 = (torch.randn(E, 2 * I, K, generator=g) * 0.05).to(torch.bfloat16).to(DEV)
    w2 = (torch.randn(E, K, I, generator=g) * 0.05).to(torch.bfloat16).to(DEV)
    wq = B.prepare_moe_weights(w1, w2)
    offsets = torch.tensor([0, 100, 100, M], dtype=torch.int32, device=DEV)
    a_codes = torch.zeros((a_rows, K // 2), dtype=torch.uint8, device=DEV)
    a_sf = torch.zeros(B.nvfp4_sf_bytes(a_rows, K, B.NVFP4_SF_TILED_ROWS), dtype=torch.uint8, device=DEV)
    row_src = torch.full((a_rows,), -1, dtype=torch.int32, device=DEV)
    row_src[:100] = torch.arange(0, 100, dtype=torch.int32, device=DEV)          # group 0 at padded row 0
    row_src[128:128 + 233] = torch.arange(100, M, dtype=torch.int32, device=DEV)  # group 2 at padded row 128
    B.nvfp4_quantize(x, row_src=row_src, codes=a_codes, sf=a_sf, gs_out=gs.view(torch.float32, (1,)),
                     sf_layout=B.NVFP4_SF_TILED_ROWS)
    gsx = gs.view(torch.float32, (1,)).clone()
    c = Guarded(M * N * 2)
    ins = {"a_codes": a_codes, "a_sf": a_sf, "w1_codes": wq["w1_codes"], "offsets": offsets}
    before = [t.clone() for t in ins.values()]
    B.nvfp4_grouped_gemm(a_codes, a_sf, gsx, wq["w1_codes"], wq["w1_sf"], wq["gs_w1"], offsets,
                         out=c.view(torch.bfloat16, (M, N)))
    _check({"c": c}, ins, before)
    hc = Guarded(a_rows * I // 2, fill=0)
    hs = Guarded(B.nvfp4_sf_bytes(a_rows, I, B.NVFP4_SF_TILED_ROWS), fill=0)
    gs_h = torch.tensor([200.0], device=DEV)
    B.nvfp4_grouped_gemm_swiglu(a_codes, a_sf, gsx, wq["w1_codes"], wq["w1_sf"], wq["gs_w1"], offsets, gs_h,
                                h_codes=hc.view(torch.uint8, (a_rows, I // 2)), h_sf=hs.view(torch.uint8, (-1,)))
    _check({"h_codes": hc, "h_sf": hs}, ins, before)
    # linear with a strided output view inside a guarded buffer
    lin = Guarded(M * (N + 8) * 2)
    lws = Guarded(int(B.lib().nvfp4_linear_workspace_size()))
    xq = torch.zeros((-(-M // 128) * 128, K // 2), dtype=torch.uint8, device=DEV)
    xs = torch.zeros(B.nvfp4_sf_bytes(xq.shape[0], K, B.NVFP4_SF_TILED_ROWS), dtype=torch.uint8, device=DEV)
    B.nvfp4_quantize(x, codes=xq[:M], sf=xs, gs_out=gs.view(torch.float32, (1,)), sf_layout=B.NVFP4_SF_TILED_ROWS)
    B.nvfp4_linear(xq, xs, gs.view(torch.float32, (1,)).clone(), M, wq["w1_codes"][0],
                   wq["w1_sf"][: B.nvfp4_sf_bytes(N, K)], wq["gs_w1"][:1],
                   out=lin.view(torch.bfloat16, (M, N + 8))[:, :N], ws=lws.bytes())
    _check({"linear": lin, "linear ws": lws}, {"x": x}, [x_in])
    # fused norm + rope + quant
    R, P = 64, 50
    xr = torch.randn(M, 192, generator=g).to(torch.bfloat16).to(DEV)
    gamma = torch.ones(192, device=DEV)
    ang = torch.rand(P, R // 2, generator=g)
    cos_t, sin_t = torch.cos(ang).to(DEV), torch.sin(ang).to(DEV)
    pos = torch.randint(0, P, (M,), generator=g, dtype=torch.int32).to(DEV)
    nc = Guarded(M * 96)
    ns = Guarded(B.nvfp4_sf_bytes(M, 192))
    ny = Guarded(M * 192 * 4)
    ins = {"x": xr, "pos": pos, "cos": cos_t, "sin": sin_t}
    before = [t.clone() for t in ins.values()]
    B.nvfp4_rmsnorm_rope_quantize(xr, gamma, 1e-6, R, pos, cos_t, sin_t, torch.tensor([100.0], device=DEV),
                                  y_out=ny.view(torch.float32, (M, 192)), codes=nc.view(torch.uint8, (M, 96)),
                                  sf=ns.view(torch.uint8, (-1,)))
    _check({"codes": nc, "sf": ns, "y": ny}, ins, before)


def test_permute_and_combine_write_only_their_outputs():
    T, k, E, K = 777, 6, 50, 256
    g = torch.Generator(device="cpu").manual_seed(10)
    ids = torch.randint(0, E, (T, k), generator=g, dtype=torch.int32).to(DEV)
    off = Guarded((E + 1) * 4)
    p2f = Guarded(T * k * 4)
    f2p = Guarded(T * k * 4)
    ws = Guarded(int(B.lib().moe_permute_workspace_size(T, k, E)))
    B.lib().moe_permute(B._ptr(ids), T, k, E, B._ptr(off.bytes()), B._ptr(p2f.bytes()), B._ptr(f2p.bytes()),
                        B._ptr(ws.bytes()), ws.n, B._stream())
    _check({"offsets": off, "p2f": p2f, "f2p": f2p, "ws": ws}, {"ids": ids}, [ids.clone()])
    out = torch.randn(T * k, K, generator=g).to(torch.bfloat16).to(DEV)
    w = torch.rand(T, k, generator=g).to(DEV)
    y = Guarded(T * K * 2)
    B.moe_combine(out, w, f2p.view(torch.int32, (T * k,)), y=y.view(torch.bfloat16, (T, K)))
    _check({"y": y}, {"out": out, "w": w}, [out.clone(), w.clone()])


def test_route_and_quantize_dispatch_write_only_their_outputs():
    """The separate stage-1/2 kernels moe_forward uses above 65536 routed rows:
    routing, then the quantize + scatter into padded rows (with the global
    scale computed), each into guarded outputs."""
    T, K, E, k = 513, 1024, 40, 6
    g = torch.Generator(device="cpu").manual_seed(12)
    x = torch.randn(T, K, generator=g).to(torch.bfloat16).to(DEV)
    logits = torch.randn(T, E, generator=g).to(DEV)
    ids = Guarded(T * k * 4)
    w = Guarded(T * k * 4)
    L = B.lib()
    assert L.moe_route_topk(B._ptr(logits), T, E, k, B._ptr(ids.bytes()), B._ptr(w.bytes()), B._stream()) == 0
    _check({"ids": ids, "w": w}, {"logits": logits}, [logits.clone()])
    offsets, p2f, f2p = B.moe_permute(ids.view(torch.int32, (T, k)), E)
    a_rows = B.nvfp4moe_padded_rows(T * k, E)
    codes = Guarded(a_rows * K // 2)
    sf = Guarded(B.nvfp4_sf_bytes(a_rows, K, B.NVFP4_SF_TILED_ROWS))
    gs = Guarded(4)
    ws = Guarded(int(L.moe_quantize_dispatch_workspace_size(E)))
    inputs = {"x": x, "offsets": offsets, "f2p": f2p}
    before = [t.clone() for t in inputs.values()]
    assert L.moe_quantize_dispatch(B._ptr(x), T, K, K, k, E, B._ptr(ids.bytes()), B._ptr(offsets), B._ptr(f2p),
                                   None, B._ptr(gs.bytes()), B._ptr(codes.bytes()), B._ptr(sf.bytes()), a_rows,
                                   B._ptr(ws.bytes()), ws.n, B._stream()) == 0
    _check({"codes": codes, "sf": sf, "gs": gs, "ws": ws}, inputs, before)
