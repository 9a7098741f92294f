"""Pins for the fp64 CPU oracle: checks against facts fixed outside the oracle itself.

Every pin takes an oracle handle so that tests/test_oracle_mutants.py can run the same
pins against deliberately broken copies of the oracle and show that each plausible
mistake is caught.

  pin_golden        hand-derived values (tests/golden/*.json, each with its citation;
                    forward out and lse, and for one file the backward dq, dk, dv)
  pin_dense         all blocks selected, full blocks -> textbook softmax attention:
                    torch's scaled_dot_product_attention and logsumexp in fp64
  pin_bruteforce    tiny inputs, an independent pure-Python enumeration that decides
                    "is key j attended by row i" by a linear scan of the LUT row, with
                    poisoned padding, out-of-range entries, clamped counts, duplicates
                    and zero / partial variable_block_sizes
  pin_invariants    softmax weights sum to one; the lse definition under another shift
  pin_closed_forms  equal keys -> mean of V and lse = log2|A| + s*log2(e);
                    constant V -> that constant; a single attended key -> v_j exactly
  pin_empty         empty rows: +0.0 (sign bit clear) and the finite sentinel
  pin_encodings     LUT -> bitmap -> attention is bit-identical to LUT -> attention;
                    bitmap <-> LUT conversions against Python set arithmetic
  pin_backward      dq, dk, dv equal fp64 torch autograd: of scaled_dot_product_attention
                    on group-repeated K/V (dense, Sq != Sk), and of a masked softmax
                    written with torch.where over a token mask built by scanning the LUT
                    (tail masks, empty rows, per-head selections)
  pin_backward_closed_forms
                    every row attends one key -> p = 1, dS = 0: dq = dk = 0 exactly and
                    dv_j = the sum of the dout rows (over the group) attending key j;
                    adding one vector to every key moves each row's scores by a constant,
                    which leaves dq, dk and dv unchanged (the D term makes each row of
                    dS sum to zero)
  pin_gqa_cross     grouped-query heads (Hq = 3 Hkv) and Sq != Sk: dense selection equals
                    fp64 scaled_dot_product_attention on K/V repeated per group; a tiny
                    per-head sparse case equals the brute-force enumeration on the
                    key/value head that each query head reads
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle as orc

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
LOG2E = 1.0 / math.log(2.0)


def _bf16_bits(x) -> np.ndarray:
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _rand_bits(shape, seed, mul=1.0):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(shape, generator=g) * mul).to(torch.bfloat16)
    return x.view(torch.int16).numpy().view(np.uint16)


# ----------------------------------------------------------------------------------
def pin_golden(h):
    for name in sorted(os.listdir(GOLDEN)):
        if not name.endswith(".json"):
            continue
        case = json.load(open(os.path.join(GOLDEN, name)))
        q = _bf16_bits(case["q"])[None, None]
        k = _bf16_bits(case["k"])[None, None]
        v = _bf16_bits(case["v"])[None, None]
        idx = np.array(case["q2k_idx"], np.int32)[None, None]
        num = np.array(case["q2k_num"], np.int32)[None, None]
        vbs = np.array(case["vbs"], np.int32)
        block = case["block"]
        out, lse = orc.vsa_forward(q, k, v, idx, num, vbs, block, math.log(2.0), h=h)
        out = out.reshape(-1, q.shape[-1])
        lse = lse.reshape(-1)
        want_out = np.array(case["out"], np.float64)
        want_lse = np.array([orc.LSE_EMPTY if x == "EMPTY" else x for x in case["lse"]])
        assert np.max(np.abs(out - want_out)) <= 1e-12, (name, out, want_out)
        assert np.max(np.abs(lse - want_lse)) <= 1e-12, (name, lse, want_lse)
        if "dout" in case:  # a backward example
            do = _bf16_bits(case["dout"])[None, None]
            grads = orc.vsa_backward(q, k, v, do, idx, num, vbs, block, math.log(2.0), h=h)
            for key, got in zip(("dq", "dk", "dv"), grads):
                want = np.array(case[key], np.float64)
                got = got.reshape(want.shape)
                assert np.max(np.abs(got - want)) <= 1e-12, (name, key, got, want)


def pin_dense(h):
    for (B, H, S, D, block, seed) in [(2, 3, 96, 16, 16, 1), (1, 2, 256, 128, 64, 2)]:
        nb = S // block
        q, k, v = (_rand_bits((B, H, S, D), seed + i) for i in range(3))
        idx = np.broadcast_to(np.arange(nb, dtype=np.int32), (B, H, nb, nb)).copy()
        num = np.full((B, H, nb), nb, np.int32)
        vbs = np.full(nb, block, np.int32)
        scale = 1.0 / math.sqrt(D)
        out, lse = orc.vsa_forward(q, k, v, idx, num, vbs, block, scale, h=h)
        out = out.reshape(B, H, S, D)
        lse = lse.reshape(B, H, S)
        tq, tk, tv = (torch.from_numpy(_bits_to_f64(x)) for x in (q, k, v))
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale)
        ref_lse = torch.logsumexp(scale * tq @ tk.transpose(-1, -2), dim=-1) / math.log(2.0)
        assert np.max(np.abs(out - ref.numpy())) <= 1e-12
        assert np.max(np.abs(lse - ref_lse.numpy())) <= 1e-12


def _brute_row(qf, kf, vf, i, block, idx_row, num, max_kv, vbs, scale):
    """Independent enumeration for one query row: for every key j decide attendance by
    scanning the LUT row slot by slot (no mask array), then softmax with math.fsum."""
    nb = len(vbs)
    n = min(max(num, 0), max_kv)
    att = []
    for j in range(kf.shape[0]):
        kb = j // block
        listed = False
        for s in range(n):
            if idx_row[s] == kb:
                listed = True
        if listed and (j - kb * block) < vbs[kb] and 0 <= kb < nb:
            att.append(j)
    if not att:
        return None, None
    s = [scale * math.fsum(qf[i, d] * kf[j, d] for d in range(kf.shape[1])) for j in att]
    m = max(s)
    w = [math.exp(x - m) for x in s]
    l = math.fsum(w)
    o = [math.fsum(w[a] * vf[att[a], d] for a in range(len(att))) / l for d in range(vf.shape[1])]
    return np.array(o), (m + math.log(l)) * LOG2E


def pin_bruteforce(h):
    rng = np.random.default_rng(7)
    for (S, D, block, max_kv) in [(48, 4, 8, 4), (64, 8, 16, 6), (40, 3, 8, 7)]:
        B, H = 2, 2
        nb = S // block
        q, k, v = (_rand_bits((B, H, S, D), 100 + S + i, mul=1.5) for i in range(3))
        idx = rng.integers(-2, nb + 2, size=(B, H, nb, max_kv)).astype(np.int32)
        # counts over the whole range, including negative and above max_kv
        num = rng.integers(-1, max_kv + 3, size=(B, H, nb)).astype(np.int32)
        num[0, 0, 0] = 0
        num[0, 0, 1] = max_kv
        idx[0, 0, 1, :] = 0          # duplicates of one block
        vbs = rng.integers(0, block + 1, size=nb).astype(np.int32)
        vbs[0] = block
        vbs[-1] = 0
        out, lse = orc.vsa_forward(q, k, v, idx, num, vbs, block, 0.37, h=h)
        out = out.reshape(B, H, S, D)
        lse = lse.reshape(B, H, S)
        qf, kf, vf = (_bits_to_f64(x) for x in (q, k, v))
        for b in range(B):
            for hh in range(H):
                for i in range(S):
                    qb = i // block
                    o, l = _brute_row(qf[b, hh], kf[b, hh], vf[b, hh], i, block,
                                      idx[b, hh, qb], int(num[b, hh, qb]), max_kv, vbs, 0.37)
                    if o is None:
                        assert np.all(out[b, hh, i] == 0.0) and lse[b, hh, i] == orc.LSE_EMPTY
                    else:
                        assert np.max(np.abs(out[b, hh, i] - o)) <= 1e-12
                        assert abs(lse[b, hh, i] - l) <= 1e-12


def pin_invariants(h):
    B, H, S, D, block = 1, 2, 128, 32, 16
    nb = S // block
    q, k = (_rand_bits((B, H, S, D), 300 + i, mul=2.0) for i in range(2))
    ones = _bf16_bits(np.ones((B, H, S, D)))
    rng = np.random.default_rng(3)
    idx = np.stack([np.stack([np.stack([rng.permutation(nb)[:5] for _ in range(nb)])
                              for _ in range(H)]) for _ in range(B)]).astype(np.int32)
    num = rng.integers(1, 6, size=(B, H, nb)).astype(np.int32)
    vbs = rng.integers(1, block + 1, size=nb).astype(np.int32)
    scale = 0.21
    out, lse = orc.vsa_forward(q, k, ones, idx, num, vbs, block, scale, h=h)
    # softmax weights sum to one: with V = 1 every output element is that sum
    assert np.max(np.abs(out - 1.0)) <= 1e-12
    # lse definition, recomputed with a different shift (c = 0 and c = 50)
    qf, kf = _bits_to_f64(q), _bits_to_f64(k)
    lse = lse.reshape(B, H, S)
    for hh in range(H):
        for i in range(0, S, 7):
            qb = i // block
            sel = set(int(x) for x in idx[0, hh, qb, :num[0, hh, qb]])
            js = [j for j in range(S) if j // block in sel and j % block < vbs[j // block]]
            s = [scale * float(np.dot(qf[0, hh, i], kf[0, hh, j])) for j in js]
            for c in (0.0, 50.0):
                want = (c + math.log(math.fsum(math.exp(x - c) for x in s))) * LOG2E
                assert abs(lse[0, hh, i] - want) <= 1e-12


def pin_closed_forms(h):
    B, H, S, D, block = 1, 1, 64, 16, 16
    nb = S // block
    rng = np.random.default_rng(11)
    q = _rand_bits((B, H, S, D), 400)
    vrand = _rand_bits((B, H, S, D), 401)
    krow = _rand_bits((D,), 402)
    kconst = np.broadcast_to(krow, (B, H, S, D)).copy()
    idx = np.full((B, H, nb, 3), -1, np.int32)
    idx[0, 0, :, 0] = [1, 0, 3, 2]
    idx[0, 0, :, 1] = [2, 3, -1, 0]
    num = np.array([[[2, 2, 1, 2]]], np.int32)
    vbs = np.array([16, 5, 9, 1], np.int32)
    scale = 0.5
    # all keys equal -> uniform weights: out = mean of V over A_i, lse = log2|A_i| + s*log2 e
    out, lse = orc.vsa_forward(q, kconst, vrand, idx, num, vbs, block, scale, h=h)
    out = out.reshape(S, D)
    lse = lse.reshape(S)
    qf, kf, vf = _bits_to_f64(q[0, 0]), _bits_to_f64(krow), _bits_to_f64(vrand[0, 0])
    for i in range(S):
        qb = i // block
        blocks = [int(x) for x in idx[0, 0, qb, :num[0, 0, qb]]]
        js = [j for b in sorted(set(blocks)) for j in range(b * block, b * block + vbs[b])]
        mean = np.array([math.fsum(vf[j, d] for j in js) / len(js) for d in range(D)])
        s = scale * math.fsum(qf[i, d] * kf[d] for d in range(D))
        assert np.max(np.abs(out[i] - mean)) <= 1e-12
        assert abs(lse[i] - (math.log2(len(js)) + s * LOG2E)) <= 1e-12
    # constant V -> that constant
    c = _bf16_bits(np.full((B, H, S, D), -2.75))
    out, _ = orc.vsa_forward(q, vrand, c, idx, num, vbs, block, scale, h=h)
    assert np.max(np.abs(out - (-2.75))) <= 1e-12
    # exactly one attended key -> v_j exactly (weight exp(0)/exp(0))
    idx1 = np.full((B, H, nb, 1), -1, np.int32)
    idx1[0, 0, :, 0] = [3, 3, 0, 1]
    vbs1 = np.array([1, 1, 1, 1], np.int32)
    num1 = np.ones((B, H, nb), np.int32)
    out, lse = orc.vsa_forward(q, vrand, vrand, idx1, num1, vbs1, block, scale, h=h)
    out = out.reshape(S, D)
    for i in range(S):
        j = int(idx1[0, 0, i // block, 0]) * block
        assert np.array_equal(out[i], vf[j])


def pin_empty(h):
    B, H, S, D, block = 1, 2, 64, 8, 16
    nb = S // block
    q, k, v = (_rand_bits((B, H, S, D), 500 + i) for i in range(3))
    idx = np.zeros((B, H, nb, 2), np.int32)
    idx[..., 1] = 3
    num = np.array([[[0, 2, 1, 2], [2, -4, 2, 0]]], np.int32)
    vbs = np.array([0, 16, 16, 0], np.int32)     # blocks 0 and 3 have no valid key
    out, lse = orc.vsa_forward(q, k, v, idx, num, vbs, block, 0.3, h=h)
    out = out.reshape(B, H, nb, block, D)
    lse = lse.reshape(B, H, nb, block)
    # every row selects only blocks {0} or {0, 3}, all with zero valid keys, or nothing
    assert np.all(out == 0.0) and not np.any(np.signbit(out))
    assert np.all(lse == orc.LSE_EMPTY)
    assert orc.LSE_EMPTY == -3.4028234663852886e38


def pin_encodings(h):
    rng = np.random.default_rng(5)
    nb, max_kv = 12, 5
    rows = 40
    idx = rng.integers(-3, nb + 3, size=(rows, max_kv)).astype(np.int32)
    num = rng.integers(-2, max_kv + 3, size=rows).astype(np.int32)
    mask = orc.lut_to_blockmask(idx, num, nb, h=h)
    for r in range(rows):
        n = min(max(int(num[r]), 0), max_kv)
        want = {int(x) for x in idx[r, :n] if 0 <= x < nb}
        got = {kb for kb in range(nb) if mask[r, kb]}
        assert got == want and set(np.unique(mask[r])) <= {0, 1}
    for cap in (nb, 3):
        li, ln = orc.blockmask_to_lut(mask, cap, h=h)
        for r in range(rows):
            want = sorted(kb for kb in range(nb) if mask[r, kb])[:cap]
            assert ln[r] == len(want)
            assert list(li[r, :ln[r]]) == want and np.all(li[r, ln[r]:] == -1)
    # any nonzero byte is "attend"
    odd = mask.astype(np.int16) * rng.integers(1, 127, size=mask.shape)
    li2, ln2 = orc.blockmask_to_lut(odd.astype(np.int8), nb, h=h)
    li1, ln1 = orc.blockmask_to_lut(mask, nb, h=h)
    assert np.array_equal(li1, li2) and np.array_equal(ln1, ln2)
    # LUT (shared by every head) -> bitmap -> Jenga forward == VSA forward, bit for bit
    B, H, S, D, block = 2, 2, 96, 16, 8
    nbq = S // block
    q, k, v = (_rand_bits((B, H, S, D), 600 + i) for i in range(3))
    idx = rng.integers(-1, nbq + 1, size=(nbq, 7)).astype(np.int32)
    num = rng.integers(0, 8, size=nbq).astype(np.int32)
    bitmap = orc.lut_to_blockmask(idx, num, nbq, h=h)
    full_idx = np.broadcast_to(idx, (B, H, nbq, 7)).copy()
    full_num = np.broadcast_to(num, (B, H, nbq)).copy()
    o1, l1 = orc.vsa_forward(q, k, v, full_idx, full_num, None, block, 0.25, h=h)
    o2, l2 = orc.jenga_forward(q, k, v, bitmap, block, 0.25, h=h)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # ... and the round trip LUT -> bitmap -> LUT -> attention is bit-identical too
    ri, rn = orc.blockmask_to_lut(bitmap, nbq, h=h)
    o3, l3 = orc.vsa_forward(q, k, v, np.broadcast_to(ri, (B, H, nbq, nbq)).copy(),
                             np.broadcast_to(rn, (B, H, nbq)).copy(), None, block, 0.25, h=h)
    assert np.array_equal(o1, o3) and np.array_equal(l1, l3)
    # a shuffled LUT row is the same set, so the same result bit for bit
    perm = rng.permutation(7)
    o4, l4 = orc.vsa_forward(q, k, v, full_idx[..., perm], full_num, None, block, 0.25, h=h)
    sel_ok = np.all(num >= 7)  # a permutation moves entries across the count boundary otherwise
    if sel_ok:
        assert np.array_equal(o1, o4)


def pin_gqa_cross(h):
    # dense: every block selected, full blocks -> textbook attention with K/V heads
    # repeated group-wise (query head hq reads key/value head hq // group)
    B, Hq, Hkv, Sq, Sk, D, block = 2, 6, 2, 64, 160, 16, 16
    nbq, nbk = Sq // block, Sk // block
    q = _rand_bits((B, Hq, Sq, D), 801)
    k, v = (_rand_bits((B, Hkv, Sk, D), 802 + i) for i in range(2))
    idx = np.broadcast_to(np.arange(nbk, dtype=np.int32), (B, Hq, nbq, nbk)).copy()
    num = np.full((B, Hq, nbq), nbk, np.int32)
    scale = 0.29
    out, lse = orc.vsa_forward(q, k, v, idx, num, None, block, scale, h=h)
    out = out.reshape(B, Hq, Sq, D)
    lse = lse.reshape(B, Hq, Sq)
    tq, tk, tv = (torch.from_numpy(_bits_to_f64(x)) for x in (q, k, v))
    tk = tk.repeat_interleave(Hq // Hkv, dim=1)
    tv = tv.repeat_interleave(Hq // Hkv, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale)
    ref_lse = torch.logsumexp(scale * tq @ tk.transpose(-1, -2), dim=-1) / math.log(2.0)
    assert np.max(np.abs(out - ref.numpy())) <= 1e-12
    assert np.max(np.abs(lse - ref_lse.numpy())) <= 1e-12
    # sparse, per-head LUT over the key blocks, tail masks, more key than query blocks
    rng = np.random.default_rng(11)
    B, Hq, Hkv, Sq, Sk, D, block, max_kv = 1, 4, 2, 24, 56, 4, 8, 5
    nbq, nbk = Sq // block, Sk // block
    q = _rand_bits((B, Hq, Sq, D), 811, mul=1.5)
    k, v = (_rand_bits((B, Hkv, Sk, D), 812 + i, mul=1.5) for i in range(2))
    idx = rng.integers(-1, nbk + 1, size=(B, Hq, nbq, max_kv)).astype(np.int32)
    num = rng.integers(0, max_kv + 1, size=(B, Hq, nbq)).astype(np.int32)
    num[0, 1, 0] = 0
    vbs = rng.integers(0, block + 1, size=nbk).astype(np.int32)
    vbs[nbk - 1] = 3
    out, lse = orc.vsa_forward(q, k, v, idx, num, vbs, block, 0.41, h=h)
    out = out.reshape(B, Hq, Sq, D)
    lse = lse.reshape(B, Hq, Sq)
    qf, kf, vf = (_bits_to_f64(x) for x in (q, k, v))
    for hq in range(Hq):
        hk = hq // (Hq // Hkv)
        for i in range(Sq):
            qb = i // block
            o, l = _brute_row(qf[0, hq], kf[0, hk], vf[0, hk], i, block, idx[0, hq, qb],
                              int(num[0, hq, qb]), max_kv, vbs, 0.41)
            if o is None:
                assert np.all(out[0, hq, i] == 0.0) and lse[0, hq, i] == orc.LSE_EMPTY
            else:
                assert np.max(np.abs(out[0, hq, i] - o)) <= 1e-12
                assert abs(lse[0, hq, i] - l) <= 1e-12


def _token_mask(idx, num, vbs, B, H, Sq, Sk, block, max_kv):
    """[B,H,Sq,Sk] bool by scanning each LUT row slot by slot (no block-mask array)."""
    m = np.zeros((B, H, Sq, Sk), dtype=bool)
    for b in range(B):
        for hh in range(H):
            for i in range(Sq):
                qb = i // block
                n = min(max(int(num[b, hh, qb]), 0), max_kv)
                for s in range(n):
                    kb = int(idx[b, hh, qb, s])
                    if 0 <= kb < Sk // block:
                        m[b, hh, i, kb * block:kb * block + int(vbs[kb])] = True
    return m


def pin_backward(h):
    # dense: all blocks, full, grouped heads, Sq != Sk -> autograd of SDPA
    B, Hq, Hkv, Sq, Sk, D, block = 1, 4, 2, 32, 48, 8, 8
    q = _rand_bits((B, Hq, Sq, D), 901)
    k, v = (_rand_bits((B, Hkv, Sk, D), 902 + i) for i in range(2))
    do = _rand_bits((B, Hq, Sq, D), 905)
    nbq, nbk = Sq // block, Sk // block
    idx = np.broadcast_to(np.arange(nbk, dtype=np.int32), (B, Hq, nbq, nbk)).copy()
    num = np.full((B, Hq, nbq), nbk, np.int32)
    scale = 0.31
    dq, dk, dv = orc.vsa_backward(q, k, v, do, idx, num, None, block, scale, h=h)
    tq, tk, tv, tdo = (torch.from_numpy(_bits_to_f64(x)) for x in (q, k, v, do))
    tq.requires_grad_(); tk.requires_grad_(); tv.requires_grad_()
    g = Hq // Hkv
    out = torch.nn.functional.scaled_dot_product_attention(
        tq, tk.repeat_interleave(g, dim=1), tv.repeat_interleave(g, dim=1), scale=scale)
    out.backward(tdo)
    for got, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        assert np.max(np.abs(got - ref.numpy())) <= 1e-11
    # sparse: LUT with tail masks, an empty query block, per-head selections
    rng = np.random.default_rng(13)
    B, Hq, Hkv, Sq, Sk, D, block, max_kv = 1, 2, 1, 24, 40, 4, 8, 4
    nbq, nbk = Sq // block, Sk // block
    q = _rand_bits((B, Hq, Sq, D), 911, mul=1.5)
    k, v = (_rand_bits((B, Hkv, Sk, D), 912 + i, mul=1.5) for i in range(2))
    do = _rand_bits((B, Hq, Sq, D), 915)
    idx = rng.integers(-1, nbk + 1, size=(B, Hq, nbq, max_kv)).astype(np.int32)
    num = rng.integers(1, max_kv + 1, size=(B, Hq, nbq)).astype(np.int32)
    num[0, 1, 2] = 0
    vbs = rng.integers(0, block + 1, size=nbk).astype(np.int32)
    vbs[0] = block
    dq, dk, dv = orc.vsa_backward(q, k, v, do, idx, num, vbs, block, 0.43, h=h)
    mask = torch.from_numpy(_token_mask(idx, num, vbs, B, Hq, Sq, Sk, block, max_kv))
    tq, tk, tv, tdo = (torch.from_numpy(_bits_to_f64(x)) for x in (q, k, v, do))
    tq.requires_grad_(); tk.requires_grad_(); tv.requires_grad_()
    kr, vr = tk.repeat_interleave(Hq // Hkv, dim=1), tv.repeat_interleave(Hq // Hkv, dim=1)
    s_ = 0.43 * tq @ kr.transpose(-1, -2)
    mx = torch.where(mask, s_, torch.tensor(-math.inf, dtype=torch.float64)).amax(-1, keepdim=True)
    mx = torch.where(torch.isinf(mx), torch.zeros_like(mx), mx).detach()
    e = torch.where(mask, torch.exp(s_ - mx), torch.zeros_like(s_))
    l_ = e.sum(-1, keepdim=True)
    out = (e / torch.where(l_ > 0, l_, torch.ones_like(l_))) @ vr
    out.backward(tdo)
    for got, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        assert np.max(np.abs(got - ref.numpy())) <= 1e-11
    assert np.all(dq[0, 1, 16:24] == 0.0)  # the empty query block


def pin_backward_closed_forms(h):
    # one attended key per row: each query block selects one key block whose first key
    # alone is valid
    rng = np.random.default_rng(21)
    B, Hq, Hkv, S, D, block = 1, 4, 2, 32, 8, 8
    nb = S // block
    q = _rand_bits((B, Hq, S, D), 931)
    k, v = (_rand_bits((B, Hkv, S, D), 932 + i) for i in range(2))
    do = _rand_bits((B, Hq, S, D), 935)
    idx = rng.integers(0, nb, size=(B, Hq, nb, 1)).astype(np.int32)
    num = np.ones((B, Hq, nb), np.int32)
    vbs = np.ones(nb, np.int32)
    dq, dk, dv = orc.vsa_backward(q, k, v, do, idx, num, vbs, block, 0.37, h=h)
    assert np.all(dq == 0.0) and np.all(dk == 0.0)
    ref = np.zeros_like(dv)
    dof = _bits_to_f64(do)
    g = Hq // Hkv
    for hq in range(Hq):
        for qb in range(nb):
            j = int(idx[0, hq, qb, 0]) * block
            ref[0, hq // g, j] += dof[0, hq, qb * block:(qb + 1) * block].sum(axis=0)
    assert np.max(np.abs(dv - ref)) <= 1e-12 * max(1.0, np.abs(ref).max())
    # keys shifted by one vector: every row's scores move by a constant
    B, Hq, Hkv, S, D, block, max_kv = 1, 2, 1, 24, 4, 8, 3
    nb = S // block
    kq = rng.integers(-8, 9, size=(B, Hkv, S, D)) / 4.0      # exact in bf16, and so is
    shift = rng.integers(-8, 9, size=D) / 4.0               # every key plus the shift
    q = _rand_bits((B, Hq, S, D), 941)
    v = _rand_bits((B, Hkv, S, D), 942)
    do = _rand_bits((B, Hq, S, D), 943)
    idx = rng.integers(0, nb, size=(B, Hq, nb, max_kv)).astype(np.int32)
    num = rng.integers(1, max_kv + 1, size=(B, Hq, nb)).astype(np.int32)
    vbs = rng.integers(1, block + 1, size=nb).astype(np.int32)
    grads = [orc.vsa_backward(q, _bf16_bits(kk), v, do, idx, num, vbs, block, 0.5, h=h)
             for kk in (kq, kq + shift)]
    for a, b in zip(*grads):
        assert np.max(np.abs(a - b)) <= 1e-10 * max(1.0, np.abs(a).max())


PINS = [pin_golden, pin_dense, pin_bruteforce, pin_invariants, pin_closed_forms, pin_empty,
        pin_encodings, pin_gqa_cross, pin_backward, pin_backward_closed_forms]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin, oracle_lib):
    pin(oracle_lib)


def test_oracle_sampled_rows_match_full(oracle_lib):
    """Computing a subset of q-blocks gives exactly the rows of the full computation."""
    B, H, S, D, block = 2, 3, 128, 16, 16
    nb = S // block
    q, k, v = (_rand_bits((B, H, S, D), 700 + i) for i in range(3))
    rng = np.random.default_rng(9)
    idx = rng.integers(0, nb, size=(B, H, nb, 4)).astype(np.int32)
    num = rng.integers(0, 5, size=(B, H, nb)).astype(np.int32)
    vbs = rng.integers(0, block + 1, size=nb).astype(np.int32)
    out, lse = orc.vsa_forward(q, k, v, idx, num, vbs, block, 0.3, h=oracle_lib)
    sel = np.array([[1, 2, 7], [0, 0, 0], [1, 1, 3]], np.int32)
    so, sl = orc.vsa_forward(q, k, v, idx, num, vbs, block, 0.3, sel=sel, h=oracle_lib)
    allsel = orc.all_qblocks(B, H, nb)
    for t, s in enumerate(sel):
        pos = int(np.nonzero((allsel == s).all(1))[0][0])
        assert np.array_equal(so[t], out[pos]) and np.array_equal(sl[t], lse[pos])
