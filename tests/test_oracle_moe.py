"""Pins for the oracle's MoE pieces (the jp-study.kr page: 256 routed experts, 8 active per
token; activations quantised to FP8 before dispatch; the gnrental.net page: combine kept in
BF16).  Routing order and gates follow the stated readings."""
import itertools
import math

import numpy as np
import pytest
import torch

from fp8_fine_grained_16_b300 import synthetic as S


def _brute_topk(row, k):
    order = sorted(range(len(row)), key=lambda e: (-float(row[e]), e))
    return order[:k]


def test_topk_brute_force_with_ties(orc):
    g = np.random.default_rng(0)
    logits = g.integers(-3, 4, size=(40, 12)).astype(np.float32)    # many ties
    r = orc.route_topk(logits, 3)
    for t in range(40):
        assert list(r["idx"][t]) == _brute_topk(logits[t], 3)


def test_gates_softmax_of_selected(orc):
    logits = S.moe_up(with_weights=False)["logits"][:64].numpy()
    r = orc.route_topk(logits, 8)
    for t in range(64):
        sel = logits[t, r["idx"][t]].astype(np.float64)
        z = np.exp(sel - sel.max())
        assert np.allclose(r["gate"][t], z / z.sum(), rtol=2e-7, atol=0)
        assert np.all(np.diff(r["gate"][t]) <= 0)        # selected in descending logit order


def test_dispatch_layout_invariants_full_size(orc):
    logits = S.moe_up(with_weights=False)["logits"].numpy()
    T, E, k = 4096, 256, 8
    r = orc.route_topk(logits, k)
    off, src, pos, idx = r["off"], r["src_row"], r["pos"], r["idx"]
    assert off[0] == 0 and off[-1] == T * k and np.all(np.diff(off) >= 0)
    counts = np.bincount(idx.ravel(), minlength=E)
    assert np.array_equal(np.diff(off), counts)
    assert np.array_equal(np.bincount(src, minlength=T), np.full(T, k))
    for t in range(T):
        assert len(set(idx[t])) == k
    assert np.array_equal(src[pos.ravel()], np.repeat(np.arange(T), k))
    for e in range(E):
        seg = src[off[e]:off[e + 1]]
        assert np.all(np.diff(seg) > 0)                   # stable: tokens ascending
        assert np.all((idx[seg] == e).any(axis=1))            # each listed token chose e


def test_permute_commutes_with_1x128_quant(orc):
    x = S.moe_up(T=256, K=512, with_weights=False)["x"]
    logits = np.random.default_rng(1).standard_normal((256, 16)).astype(np.float32)
    r = orc.route_topk(logits, 4)
    xb = S.bf16_bits(x)
    q, s = orc.quant_act_1x128(xb)
    qp, sp = orc.permute_rows(q, s, r["src_row"])
    q2, s2 = orc.quant_act_1x128(xb[r["src_row"]])
    assert np.array_equal(qp, q2) and np.array_equal(sp, s2)


def test_grouped_equals_dense_per_expert(orc):
    g = np.random.default_rng(2)
    E, N, K = 5, 256, 256
    off = np.array([0, 3, 3, 40, 41, 60], np.int32)          # includes an empty expert
    total = int(off[-1])
    a = g.integers(0, 0x7E, size=(total, K)).astype(np.uint8)
    b = g.integers(0, 0x7E, size=(E, N, K)).astype(np.uint8)
    sa = g.uniform(0.1, 2, size=(K // 128, total)).astype(np.float32)
    sb = g.uniform(0.1, 2, size=(E, N // 128, K // 128)).astype(np.float32)
    d = orc.grouped_gemm_blockscaled(a, sa, b, sb, off)
    for e in range(E):
        lo, hi = off[e], off[e + 1]
        if lo == hi:
            continue
        de = orc.gemm_blockscaled(a[lo:hi], np.ascontiguousarray(sa[:, lo:hi]), b[e], sb[e], 0)
        assert np.array_equal(d[lo:hi], de)


def test_combine_one_hot_is_gather(orc):
    T, k, N = 50, 4, 96
    g = np.random.default_rng(3)
    y = torch.randn((T * k, N), generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    yb = S.bf16_bits(y)
    pos = np.stack([g.permutation(T * k)[:k] for _ in range(T)]).astype(np.int32)
    gate = np.zeros((T, k), np.float32)
    hot = g.integers(0, k, size=T)
    gate[np.arange(T), hot] = 1.0
    out = orc.moe_combine(yb, pos, gate)
    assert np.array_equal(out, yb[pos[np.arange(T), hot]])


def test_combine_is_rounded_weighted_sum(orc):
    T, k, N = 20, 8, 64
    y = torch.randn((T * k, N), generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    g = np.random.default_rng(4)
    pos = np.stack([g.permutation(T * k)[:k] for _ in range(T)]).astype(np.int32)
    gate = g.dirichlet(np.ones(k), size=T).astype(np.float32)
    out = orc.moe_combine(S.bf16_bits(y), pos, gate)
    yf = y.double().numpy()
    exact = np.einsum("tj,tjn->tn", gate.astype(np.float64), yf[pos])
    # one rounding of a (near-)exact fp64 sum: at most half a bf16 ulp away
    outf = S.from_bf16_bits(out).double().numpy()
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(exact), 1e-30))) - 7)
    assert np.all(np.abs(outf - exact) <= 0.5 * ulp * (1 + 1e-9))
