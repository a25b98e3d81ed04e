"""GPU parity of nvfp4_linear (the single-expert NVFP4 linear for shared
experts and projections) against the fp64 oracle, and of a shared-expert MLP
run on a side stream concurrently with the routed-expert forward."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import assert_close_tol, cosine
from nvfp4_block_scaled_05_gb300 import binding as B
from nvfp4_block_scaled_05_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _quantize_padded(x):
    """NVFP4 codes of x (M, K) in a buffer of 128*ceil(M/128) rows (the
    padding rows zero), tiled scales, device global scale."""
    M, K = x.shape
    a_rows = max(128, -(-M // 128) * 128)
    codes = torch.zeros((a_rows, K // 2), dtype=torch.uint8, device=x.device)
    sf = torch.zeros(B.nvfp4_sf_bytes(a_rows, K, B.NVFP4_SF_TILED_ROWS), dtype=torch.uint8, device=x.device)
    _, _, gs = B.nvfp4_quantize(x, codes=codes[:M], sf=sf, sf_layout=B.NVFP4_SF_TILED_ROWS)
    return codes, sf, gs


@pytest.mark.parametrize("M,N,K", [(300, 384, 512), (1, 128, 64), (128, 256, 7168)])
def test_linear_matches_oracle(M, N, K):
    g = torch.Generator(device="cpu").manual_seed(M + N + K)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    w = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16)
    ac, asf, gsa = _quantize_padded(x.to(DEV))
    wc, wsf, gsw = B.nvfp4_quantize(w.to(DEV))
    c = B.nvfp4_linear(ac, asf, gsa, M, wc, wsf, gsw)
    assert B.nvfp4moe_last_device_status() == 0
    xb, wb = W.bf16_bits(x), W.bf16_bits(w)
    g1, g2 = O.global_scale(O.amax_bf16(xb)), O.global_scale(O.amax_bf16(wb))
    assert gsa.item() == g1 and gsw.item() == g2
    ref = O.matmul_nt(O.dequantize_f64(*O.quantize_bf16(xb, g1), g1), O.dequantize_f64(*O.quantize_bf16(wb, g2), g2))
    got = c.float().cpu().numpy()
    assert_close_tol(got, ref, "linear %dx%dx%d" % (M, N, K))
    assert cosine(got, ref) > 0.9999


def _shared_expert(x, sw, gs_h):
    """Shared-expert MLP: y = W2 . swiglu(W1 . x), NVFP4 throughout (one group)."""
    T = x.shape[0]
    ac, asf, gsx = _quantize_padded(x)
    bounds = torch.tensor([0, T], dtype=torch.int32, device=x.device)
    hc, hsf = B.nvfp4_grouped_gemm_swiglu(ac, asf, gsx, sw["w1_codes"], sw["w1_sf"], sw["gs_w1"], bounds, gs_h)
    return B.nvfp4_linear(hc, hsf, gs_h, T, sw["w2_codes"][0], sw["w2_sf"], sw["gs_w2"])


def test_shared_expert_concurrent_with_routed_experts():
    cfg = W.MoEConfig("shared", T=256, K=1024, I=512, E=16, k=4, gs_h=336.0)
    inp = W.moe_inputs(cfg, seed=5, device=DEV)
    wts = B.prepare_moe_weights(inp["w1"], inp["w2"])
    g = torch.Generator(device="cpu").manual_seed(77)
    w1s = (torch.randn(1, 2 * cfg.I, cfg.K, generator=g) * 0.05).to(torch.bfloat16)
    w2s = (torch.randn(1, cfg.K, cfg.I, generator=g) * 0.05).to(torch.bfloat16)
    sw = B.prepare_moe_weights(w1s.to(DEV), w2s.to(DEV))
    gs_h = torch.tensor([cfg.gs_h], dtype=torch.float32, device=DEV)
    x, logits = inp["x"], inp["logits"]
    # sequential
    y_moe = B.moe_forward(x, logits, wts, cfg.k, gs_h).clone()
    y_sh = _shared_expert(x, sw, gs_h).clone()
    torch.cuda.synchronize()
    # concurrent: routed experts on one stream, the shared expert on another
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s1):
        y_moe2 = B.moe_forward(x, logits, wts, cfg.k, gs_h)
    with torch.cuda.stream(s2):
        y_sh2 = _shared_expert(x, sw, gs_h)
    torch.cuda.current_stream().wait_stream(s1)
    torch.cuda.current_stream().wait_stream(s2)
    torch.cuda.synchronize()
    assert B.nvfp4moe_last_device_status() == 0
    assert torch.equal(y_moe, y_moe2) and torch.equal(y_sh, y_sh2)
    # the shared expert against the oracle: one expert, top-1, weight 1
    xb = W.bf16_bits(x)
    w1b, w2b = W.bf16_bits(w1s[0]), W.bf16_bits(w2s[0])
    ref = O.moe_forward(xb, np.zeros((cfg.T, 1), np.float32), lambda e: w1b, lambda e: w2b, 1,
                        np.float32(cfg.gs_h))
    got = y_sh.float().cpu().numpy()
    assert_close_tol(got, ref["y"], "shared expert")
    assert cosine(got, ref["y"]) >= 0.9995
