"""GPU parity for the backward (vsa_bwd): dq, dk, dv against the fp64 oracle backward on the
same seeded inputs, for the forward's own out and lse.

Tolerance (no gradient tolerance is stated by the pages; derived from the arithmetic):
dq, dk, dv are written in bf16 (relative rounding 2^-9), P and dS are rounded to bf16 before
their tensor-core products, and D = dout . out uses the bf16 out -- a few 2^-9 relative
terms per element.  The test bounds, per tensor, max|gpu - oracle| <= 2e-2 * max|oracle|
and mean|gpu - oracle| <= 1.5e-2 * mean|oracle| (measured: <= 5.7e-3 and <= 6.3e-3).
"""
import numpy as np
import pytest
import torch

from block_sparse_attention_vsa_gb300 import binding, workloads
from oracle import oracle as orc

pytestmark = pytest.mark.gpu

REL_MAX, REL_MEAN = 2e-2, 1.5e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def run_and_compare(w, seed=1):
    d = torch.device("cuda:0")
    q, k, v = (t.to(d) for t in (w.q, w.k, w.v))
    idx, num, vbs = (torch.from_numpy(np.ascontiguousarray(x)).to(d)
                     for x in (w.q2k_idx, w.q2k_num, w.vbs))
    out, lse = binding.vsa_fwd_gqa(q, k, v, idx, num, vbs, block=w.block, scale=w.scale)
    g = torch.Generator().manual_seed(seed)
    do = torch.randn(w.q.shape, generator=g).to(torch.bfloat16)
    dq, dk, dv = binding.vsa_bwd(q, k, v, out, do.to(d), lse, idx, num, vbs, block=w.block,
                                 scale=w.scale)
    torch.cuda.synchronize()
    code, detail = binding.vsa_device_status()
    assert code == binding.VSA_OK, hex(detail)
    refs = orc.vsa_backward(workloads.bits(w.q), workloads.bits(w.k), workloads.bits(w.v),
                            workloads.bits(do), w.q2k_idx, w.q2k_num, w.vbs, w.block, w.scale)
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        got = got.float().cpu().numpy().astype(np.float64)
        e = np.abs(got - ref)
        scale_max, scale_mean = np.abs(ref).max(), np.abs(ref).mean()
        if scale_max == 0.0:
            assert np.all(got == 0.0), name
            continue
        assert e.max() <= REL_MAX * scale_max, (name, e.max(), scale_max)
        assert e.mean() <= REL_MEAN * scale_mean, (name, e.mean(), scale_mean)
    return dq, dk, dv


@pytest.mark.parametrize("block", [64, 128])
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (4, 1), (6, 2)])
def test_backward_matches_oracle(block, Hq, Hkv):
    w = workloads.make_random_gqa(1, Hq, Hkv, 6 * block, 8 * block, 128, block, 5,
                                  seed=120 + Hq + Hkv, vbs_lo=0, vbs_hi=block)
    run_and_compare(w)


@pytest.mark.parametrize("block", [64, 128])
def test_backward_cross_length_and_empty_rows(block):
    w = workloads.make_random_gqa(2, 2, 1, 3 * block, 11 * block, 128, block, 6, seed=130,
                                  vbs_lo=0, vbs_hi=block)
    w.q2k_num[0, 1, :] = 0      # a query head that attends nothing
    w.q2k_num[1, 0, 2] = 0      # one empty query block
    dq, dk, dv = run_and_compare(w)
    assert torch.count_nonzero(dq[0, 1]).item() == 0


def test_backward_peaky_and_dense():
    run_and_compare(workloads.make_random_gqa(1, 2, 1, 256, 1024, 128, 64, 12, seed=131,
                                              n_lo=4, qk_mul=3.0))
    run_and_compare(workloads.make_random_gqa(1, 2, 2, 512, 512, 128, 64, 8, seed=132, n_lo=8))


def test_backward_unattended_keys_get_zero():
    # every query block takes only key block 0: all other dk, dv are exactly zero
    w = workloads.make_random_gqa(1, 2, 2, 256, 512, 128, 64, 1, seed=133, n_lo=1)
    w.q2k_idx[...] = 0
    dq, dk, dv = run_and_compare(w)
    assert torch.count_nonzero(dk[:, :, 64:]).item() == 0
    assert torch.count_nonzero(dv[:, :, 64:]).item() == 0


def test_backward_no_query_rows_zeroes_dk_dv():
    d = torch.device("cuda:0")
    k = torch.randn(1, 2, 256, 128, device=d).to(torch.bfloat16)
    v = torch.randn_like(k)
    q = torch.empty(1, 2, 0, 128, dtype=torch.bfloat16, device=d)
    idx = torch.zeros(1, 2, 0, 4, dtype=torch.int32, device=d)
    num = torch.zeros(1, 2, 0, dtype=torch.int32, device=d)
    lse = torch.empty(1, 2, 0, dtype=torch.float32, device=d)
    dq, dk, dv = binding.vsa_bwd(q, k, v, q, q, lse, idx, num, None, block=64)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dk).item() == 0 and torch.count_nonzero(dv).item() == 0


def test_backward_larger_case():
    # 8 heads of 4096 queries, 64 blocks, 16 of them selected per query block
    w = workloads.make_random_gqa(1, 8, 4, 4096, 4096, 128, 64, 16, seed=134, n_lo=16,
                                  vbs_lo=48, vbs_hi=64)
    run_and_compare(w)


def test_backward_column_longer_than_one_list_chunk():
    # 8 query heads share one key/value head and all 512 query blocks of each select key
    # blocks 0 and 1: 4096 (head, query block) pairs select each of them, more than one
    # 2048-entry list chunk
    w = workloads.make_random_gqa(1, 8, 1, 512 * 64, 4 * 64, 128, 64, 2, seed=135, n_lo=2)
    w.q2k_idx[..., 0] = 0
    w.q2k_idx[..., 1] = 1
    run_and_compare(w)


@pytest.mark.parametrize("block", [64, 128])
def test_backward_odd_column_lengths(block):
    """Key blocks selected by 1, 3, 0 and 5 query blocks (of 6, two query heads sharing a
    key/value head, so 2, 6, 0, 10 entries; and 1, 3, 0, 5 with one head).  With block 64
    the key tile pairs blocks 0 and 1 (whose query blocks partly differ, so entries select
    one or both) and blocks 2 and 3, where block 2, which nobody selects, shares the tile
    with block 3; a key block nobody selects gets dk = dv = 0."""
    for hq in (1, 2):
        w = workloads.make_random_gqa(1, hq, 1, 6 * block, 4 * block, 128, block, 4,
                                      seed=140 + hq, vbs_lo=block // 2, vbs_hi=block)
        sel = {0: [2], 1: [0, 3, 5], 2: [], 3: [0, 1, 2, 4, 5]}
        w.q2k_idx[...] = -1
        w.q2k_num[...] = 0
        for kb, qbs in sel.items():
            for qb in qbs:
                for h in range(hq):
                    n = w.q2k_num[0, h, qb]
                    w.q2k_idx[0, h, qb, n] = kb
                    w.q2k_num[0, h, qb] = n + 1
        dq, dk, dv = run_and_compare(w)
        rows = slice(2 * block, 3 * block)
        assert not dk[0, 0, rows].float().abs().any() and not dv[0, 0, rows].float().abs().any()



def test_backward_block64_pairs_one_sided_and_lone_last_block():
    """Block 64 runs key blocks in adjacent pairs.  Five key blocks (the last pair is a lone
    block whose partner rows lie past the end of the keys): pair (0, 1) has query blocks
    selecting only block 0, only block 1 and both; in pair (2, 3) only block 3 is selected;
    the lone block 4 is selected with a 40-key tail.  Two query heads share a key/value
    head, so a column mixes heads."""
    w = workloads.make_random_gqa(1, 2, 1, 6 * 64, 5 * 64, 128, 64, 4, seed=151,
                                  vbs_lo=64, vbs_hi=64)
    w.vbs[4] = 40
    sel = {0: [0, 2], 1: [1, 2, 5], 2: [], 3: [0, 4], 4: [1, 3, 5]}
    w.q2k_idx[...] = -1
    w.q2k_num[...] = 0
    for kb, qbs in sel.items():
        for qb in qbs:
            for h in range(2):
                n = w.q2k_num[0, h, qb]
                w.q2k_idx[0, h, qb, n] = kb
                w.q2k_num[0, h, qb] = n + 1
    dq, dk, dv = run_and_compare(w)
    rows = slice(2 * 64, 3 * 64)  # key block 2: selected by nobody
    assert not dk[0, 0, rows].float().abs().any() and not dv[0, 0, rows].float().abs().any()
    assert not dk[0, 0, 4 * 64 + 40:].float().abs().any()  # the tail keys of block 4

def _sampled_full_size(w, samples):
    """The backward of workload ``w`` at full size, in the launch configuration the
    benchmark times, checked on sampled key blocks ``samples`` = [(b, h, kb)].  The query
    blocks selecting a key block are the only ones feeding its dk, dv, and each of their dq
    rows depends only on that row's own attention (over every key its query block selects),
    so an oracle run on just those query blocks with the head's full keys (one sub-problem
    per sample, padded with query blocks that select nothing) gives exact dk, dv for the
    key block and exact dq for every query block in its column."""
    d = torch.device("cuda:0")
    q, k, v = (t.to(d) for t in (w.q, w.k, w.v))
    idx, num, vbs = (torch.from_numpy(np.ascontiguousarray(x)).to(d)
                     for x in (w.q2k_idx, w.q2k_num, w.vbs))
    out, lse = binding.vsa_fwd_gqa(q, k, v, idx, num, vbs, block=w.block, scale=w.scale)
    do = torch.randn(w.q.shape, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    dq, dk, dv = binding.vsa_bwd(q, k, v, out, do.to(d), lse, idx, num, vbs, block=w.block,
                                 scale=w.scale)
    torch.cuda.synchronize()
    code, detail = binding.vsa_device_status()
    assert code == binding.VSA_OK, hex(detail)
    # bf16 on the host; only the sampled slices are widened below
    dq, dk, dv = (t.cpu() for t in (dq, dk, dv))
    del q, k, v, idx, num, vbs, out, lse
    wide = lambda t: t.float().numpy().astype(np.float64)

    blk, nb, D = w.block, w.nb, w.D
    mask = orc.lut_to_blockmask(w.q2k_idx, w.q2k_num, nb)  # [B, H, nb, nb]
    cols = [np.nonzero(mask[b, h, :, kb])[0] for b, h, kb in samples]
    assert all(len(c) > 0 for c in cols), "a sampled key block no query block selects"
    nmax = max(len(c) for c in cols)
    bits = {name: workloads.bits(t) for name, t in (("q", w.q), ("k", w.k), ("v", w.v),
                                                    ("do", do))}
    n = len(samples)
    qs = np.zeros((1, n, nmax * blk, D), np.uint16)
    dos = np.zeros_like(qs)
    ks = np.zeros((1, n, w.S, D), np.uint16)
    vs = np.zeros_like(ks)
    ms = np.zeros((1, n, nmax, nb), np.int8)
    for s, ((b, h, kb), col) in enumerate(zip(samples, cols)):
        for t, qb in enumerate(col):
            qs[0, s, t * blk:(t + 1) * blk] = bits["q"][b, h, qb * blk:(qb + 1) * blk]
            dos[0, s, t * blk:(t + 1) * blk] = bits["do"][b, h, qb * blk:(qb + 1) * blk]
            ms[0, s, t] = mask[b, h, qb]
        ks[0, s] = bits["k"][b, h]
        vs[0, s] = bits["v"][b, h]
    rq, rk, rv = orc.masked_attention_bwd(qs, ks, vs, dos, ms, blk, w.scale, vbs=w.vbs)

    got = {"dq": [], "dk": [], "dv": []}
    ref = {"dq": [], "dk": [], "dv": []}
    for s, ((b, h, kb), col) in enumerate(zip(samples, cols)):
        keys = slice(kb * blk, (kb + 1) * blk)
        got["dk"].append(wide(dk[b, h, keys]))
        ref["dk"].append(rk[0, s, keys])
        got["dv"].append(wide(dv[b, h, keys]))
        ref["dv"].append(rv[0, s, keys])
        for t, qb in enumerate(col):
            got["dq"].append(wide(dq[b, h, qb * blk:(qb + 1) * blk]))
            ref["dq"].append(rq[0, s, t * blk:(t + 1) * blk])
    for name in ("dq", "dk", "dv"):
        g, r = np.concatenate(got[name]), np.concatenate(ref[name])
        e = np.abs(g - r)
        assert e.max() <= REL_MAX * np.abs(r).max(), (name, e.max(), np.abs(r).max())
        assert e.mean() <= REL_MEAN * np.abs(r).mean(), (name, e.mean(), np.abs(r).mean())


def test_mid_workload_sampled_full_size():
    # vsa_mid: the first and last key blocks, neighbouring ones, several heads
    w = workloads.make("vsa_mid")
    _sampled_full_size(w, [(0, 0, 0), (0, 0, 255), (0, 5, 128), (0, 11, 63), (0, 3, 1),
                           (0, 7, 200)])


def test_blk128_workload_sampled_full_size():
    # vsa_blk128 (two batches, 24 heads, block 128, tail masks 96..128): the first and
    # last key blocks, both batches, several heads
    w = workloads.make("vsa_blk128")
    _sampled_full_size(w, [(0, 0, 0), (1, 23, 255), (0, 17, 128), (1, 4, 31), (1, 9, 200)])


def test_long_video_workload_sampled_full_size():
    # vsa_long_video (24 heads of 98,304 keys, block 64, 3-D neighbourhood selections):
    # the first key block, one in the middle of the grid and the last one, whose 32 valid
    # keys exercise the tail mask, on different heads
    w = workloads.make("vsa_long_video")
    _sampled_full_size(w, [(0, 0, 0), (0, 11, 700), (0, 23, 1535)])
