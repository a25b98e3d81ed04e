"""GPU parity of routing (top-k ids bit-exact, weights within 1e-6),
permutation (bit-exact) and combine (fp64 oracle, float tolerance)."""
import numpy as np
import pytest
import torch

import oracle as O
from nvfp4_block_scaled_05_gb300 import binding as B
from nvfp4_block_scaled_05_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "skewed"])
def test_route_topk_matches_oracle(name):
    cfg = W.CONFIGS[name]
    logits = W.moe_inputs(cfg, seed=0, weights=False)["logits"]
    ids, w = B.moe_route_topk(logits.to(DEV), cfg.k)
    torch.cuda.synchronize()
    rid, rw = O.route_topk(logits.numpy(), cfg.k)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert np.allclose(w.cpu().numpy(), rw, rtol=1e-6, atol=1e-7)


def test_route_ties_and_odd_expert_counts():
    rng = np.random.default_rng(0)
    for E, k in [(3, 3), (33, 5), (70, 16), (1024, 8)]:
        logits = rng.integers(-3, 3, (257, E)).astype(np.float32)   # many ties
        ids, w = B.moe_route_topk(torch.from_numpy(logits).to(DEV), k)
        rid, rw = O.route_topk(logits, k)
        assert np.array_equal(ids.cpu().numpy(), rid), (E, k)
        assert np.allclose(w.cpu().numpy(), rw, rtol=1e-6, atol=1e-7)


def test_route_nan_logits_decode_shape():
    """Reading R16 (a NaN logit ranks as -inf) on a decode-shaped batch (T=128,
    E=256, top-8) with NaN logits scattered over it, including rows whose
    largest logit position holds a NaN and a row with fewer than k finite
    logits: ids bit-exact against the oracle, weights within 1e-6."""
    rng = np.random.default_rng(11)
    T, E, k = 128, 256, 8
    logits = rng.normal(0, 1, (T, E)).astype(np.float32)
    logits[rng.random((T, E)) < 0.05] = np.nan
    top = np.argmax(np.nan_to_num(logits, nan=-np.inf), axis=1)
    logits[np.arange(0, T, 3), top[::3]] = np.nan          # the would-be winner is NaN
    logits[5, :] = np.nan
    logits[5, [17, 200, 3, 99, 64]] = [0.5, -1.0, 2.0, 0.0, 1.5]   # 5 finite logits, k = 8
    ids, w = B.moe_route_topk(torch.from_numpy(logits).to(DEV), k)
    torch.cuda.synchronize()
    rid, rw = O.route_topk(logits, k)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert np.allclose(w.cpu().numpy(), rw, rtol=1e-6, atol=1e-7)
    assert np.all(np.isfinite(w.cpu().numpy()))


@pytest.mark.parametrize("T,k,E,mode", [(1, 1, 1, "uniform"), (64, 2, 8, "uniform"),
                                         (128, 8, 256, "uniform"), (16384, 8, 256, "uniform"),
                                         (5000, 8, 256, "one"), (3000, 4, 1000, "sparse"),
                                         (333, 6, 384, "uniform")])
def test_permute_bit_exact(T, k, E, mode):
    rng = np.random.default_rng(T + E)
    if mode == "uniform":
        ids = rng.integers(0, E, (T, k))
    elif mode == "one":
        ids = np.full((T, k), E // 3)
    else:
        ids = rng.choice([1, 7, E - 1], (T, k))
    ids = ids.astype(np.int32)
    off, p2f, f2p = B.moe_permute(torch.from_numpy(ids).to(DEV), E)
    torch.cuda.synchronize()
    roff, rp2f, rf2p = O.permute(ids, E)
    assert np.array_equal(off.cpu().numpy(), roff)
    assert np.array_equal(p2f.cpu().numpy(), rp2f)
    assert np.array_equal(f2p.cpu().numpy(), rf2p)


def test_permute_deterministic_rerun():
    ids = torch.randint(0, 256, (16384, 8), dtype=torch.int32, generator=torch.Generator().manual_seed(3))
    a = [t.cpu() for t in B.moe_permute(ids.to(DEV), 256)]
    b = [t.cpu() for t in B.moe_permute(ids.to(DEV), 256)]
    assert all(torch.equal(x, y) for x, y in zip(a, b))


def test_combine_matches_oracle():
    rng = np.random.default_rng(5)
    T, k, K = 300, 8, 7168
    out = torch.from_numpy(rng.normal(0, 1, (T * k, K)).astype(np.float32)).to(torch.bfloat16)
    perm = rng.permutation(T * k).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    y = B.moe_combine(out.to(DEV), torch.from_numpy(w).to(DEV), torch.from_numpy(perm).to(DEV))
    torch.cuda.synchronize()
    ref = O.combine(out.float().numpy().astype(np.float64), w.astype(np.float64), perm)
    got = y.float().cpu().numpy()
    # f32 accumulation then one BF16 rounding: |err| <= 2^-8 |ref| + f32 slack
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5 * np.abs(w).sum(1, keepdims=True) * 8)
