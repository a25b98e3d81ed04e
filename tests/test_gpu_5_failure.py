"""Failure detection without a GPU fault: every wait in the GEMM kernels is
bounded. With the test stall on, the MMA-issuing thread waits on a barrier
that nothing arrives on; after the (short) wait limit the kernel records
NVFP4MOE_ERR_DEVICE_TIMEOUT in its status word, the other roles see the abort
flag, drain their own copies and tensor-core work, free the tensor memory and
return; the host reads the status and the context stays usable for the next,
normal launch."""
import numpy as np
import pytest
import torch

from nvfp4_block_scaled_05_gb300 import binding as B

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _operands():
    g = torch.Generator().manual_seed(9)
    E, K, N, per = 4, 1024, 256, 200
    M = E * per
    offsets = torch.arange(0, M + 1, per, dtype=torch.int32).to(DEV)
    a_rows = B.nvfp4moe_padded_rows(M, E)
    a_codes = torch.randint(0, 256, (a_rows, K // 2), dtype=torch.uint8, generator=g).to(DEV)
    a_sf = torch.full((B.nvfp4_sf_bytes(a_rows, K, B.NVFP4_SF_TILED_ROWS),), 0x38, dtype=torch.uint8, device=DEV)
    b_codes = torch.randint(0, 256, (E, N, K // 2), dtype=torch.uint8, generator=g).to(DEV)
    b_sf = torch.full((E * B.nvfp4_sf_bytes(N, K),), 0x38, dtype=torch.uint8, device=DEV)
    one = torch.ones(1, device=DEV)
    gsb = torch.ones(E, device=DEV)
    return a_codes, a_sf, one, b_codes, b_sf, gsb, offsets


@pytest.mark.parametrize("mode", [0, 1])
def test_wait_timeout_is_reported_and_context_survives(mode):
    """mode 0: one CTA per tile; mode 1: the 2-SM pair kernel (the even CTA's
    MMA issuer stalls; the odd CTA learns of the abort from its flag, which the
    even CTA sets remotely, and both leave through the exit handshake)."""
    ops = _operands()
    B.nvfp4moe_set_gemm_mode(mode)
    try:
        assert B.nvfp4moe_last_device_status() == 0
        good = B.nvfp4_grouped_gemm(*ops).clone()
        assert B.nvfp4moe_last_device_status() == 0
        try:
            B.nvfp4moe_set_wait_limit_ns(20_000_000)      # 20 ms
            B.nvfp4moe_set_test_stall(True)
            B.nvfp4_grouped_gemm(*ops)
            st = B.nvfp4moe_last_device_status()
        finally:
            B.nvfp4moe_set_test_stall(False)
            B.nvfp4moe_set_wait_limit_ns(4_000_000_000)
        assert st == -5
        # status was read and cleared; a normal launch still works and matches
        again = B.nvfp4_grouped_gemm(*ops)
        assert B.nvfp4moe_last_device_status() == 0
        assert torch.equal(good, again)
    finally:
        B.nvfp4moe_set_gemm_mode(0)
    assert torch.isfinite(good.float()).all()


@pytest.mark.parametrize("front,size", [("static", "tiny"), ("dynamic", "tiny"), ("static", "big"),
                                       ("dynamic", "big")])
def test_front_barrier_timeout_is_reported_and_context_survives(front, size):
    """The fused front (moe_forward_static with its given global scale, or
    moe_forward, whose dispatch computes it): with the test stall on, block 0
    leaves before the first grid barrier; the other blocks' bounded barrier
    waits run out, the status reads NVFP4MOE_ERR_DEVICE_TIMEOUT, the later
    stages find no rows, and the next normal call gives the normal result.
    "big" has more routed rows than FRONT_FUSED_QUANTIZE_MAX_ROWS, so the
    quantize + scatter runs as a second kernel after the timed-out one (on the
    zeroed offsets, positions and padded starts: every slot into row 0)."""
    from nvfp4_block_scaled_05_gb300 import workloads as W
    if size == "tiny":
        cfg = W.CONFIGS["tiny"]
    else:
        T = B.FRONT_FUSED_QUANTIZE_MAX_ROWS // 8 + 64
        cfg = W.MoEConfig("big", T=T, K=256, I=128, E=8, k=8, gs_h=1344.0)
        assert T * cfg.k > B.FRONT_FUSED_QUANTIZE_MAX_ROWS
    inp = W.moe_inputs(cfg, seed=4, device=DEV)
    wts = B.prepare_moe_weights(inp["w1"], inp["w2"])
    gs_h = torch.tensor([cfg.gs_h], dtype=torch.float32, device=DEV)
    gs_x = torch.tensor([500.0], dtype=torch.float32, device=DEV)
    if front == "static":
        fwd = lambda: B.moe_forward_static(inp["x"], inp["logits"], wts, cfg.k, gs_h, gs_x)
    else:
        assert B.moe_forward_uses_fused_dispatch(cfg.T, cfg.E, cfg.k)
        fwd = lambda: B.moe_forward(inp["x"], inp["logits"], wts, cfg.k, gs_h)
    good = fwd().clone()
    assert B.nvfp4moe_last_device_status() == 0
    try:
        B.nvfp4moe_set_wait_limit_ns(20_000_000)
        B.nvfp4moe_set_test_stall(True)
        fwd()
        st = B.nvfp4moe_last_device_status()
    finally:
        B.nvfp4moe_set_test_stall(False)
        B.nvfp4moe_set_wait_limit_ns(4_000_000_000)
    assert st == -5
    again = fwd()
    assert B.nvfp4moe_last_device_status() == 0
    assert torch.equal(good, again)
