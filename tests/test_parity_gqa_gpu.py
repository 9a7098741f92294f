"""GPU parity for grouped-query heads (Hq = g * Hkv), separate query / key lengths
(Sq != Sk), odd query-block counts and the block-map (from-mask) forward, through the C
ABI against the fp64 oracle on the same seeded inputs (tolerances in tests/gpu_util.py).

Shapes follow "TheRock rocke sparse_attention.py" (JengaSparseSpec / VsaSparseSpec:
seqlen_q, seqlen_k, query and key-value head counts) and "FastVideo
block_sparse_attn_sm100a.py" (from-mask inference: a block map per batch and head).
"""
import numpy as np
import pytest
import torch

from block_sparse_attention_vsa_gb300 import binding, workloads
from gpu_util import compare, run_gpu, sample_qblocks, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def gqa(block, seed, B=1, Hq=4, Hkv=2, nbq=6, nbk=10, max_kv=7, kind="vsa", **kw):
    return workloads.make_random_gqa(B, Hq, Hkv, nbq * block, nbk * block, 128, block, max_kv,
                                     seed, vbs_lo=0, vbs_hi=block, kind=kind, **kw)


@pytest.mark.parametrize("block", [64, 128])
@pytest.mark.parametrize("Hq,Hkv", [(4, 1), (6, 2), (8, 8)])
def test_grouped_heads(block, Hq, Hkv):
    w = gqa(block, 40 + Hq + Hkv, B=2, Hq=Hq, Hkv=Hkv, nbq=8, nbk=8)
    out, lse = run_gpu(w)
    compare(w, out, lse)


@pytest.mark.parametrize("block", [64, 128])
@pytest.mark.parametrize("nbq,nbk", [(4, 24), (24, 4), (7, 9), (1, 1), (5, 2)])
def test_cross_length(block, nbq, nbk):
    w = gqa(block, 50 + nbq * 31 + nbk, Hq=4, Hkv=2, nbq=nbq, nbk=nbk)
    out, lse = run_gpu(w)
    compare(w, out, lse)


@pytest.mark.parametrize("block", [64, 128])
def test_odd_query_blocks_write_nothing_past_the_output(block):
    # an odd number of query blocks leaves the last block-64 item with one block; its
    # second half must not be stored (the rows past Sq belong to nobody)
    w = gqa(block, 61, B=1, Hq=2, Hkv=1, nbq=3, nbk=5)
    dev = to_dev(w)
    n = w.q.numel()
    buf = torch.full((n + 64 * 128 * 2,), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = buf[:n].view_as(dev["q"])
    lbuf = torch.full((w.B * w.H * w.S + 256,), float("nan"), dtype=torch.float32, device="cuda")
    lse = lbuf[:w.B * w.H * w.S].view(w.B, w.H, w.S)
    binding.vsa_fwd_gqa(dev["q"], dev["k"], dev["v"], dev["idx"], dev["num"], dev["vbs"],
                        block=block, scale=w.scale, out=out, lse=lse)
    torch.cuda.synchronize()
    assert torch.isnan(buf[n:].float()).all(), "rows past the output were written"
    assert torch.isnan(lbuf[w.B * w.H * w.S:]).all(), "lse past the output was written"
    compare(w, out, lse)


def test_odd_query_blocks_through_vsa_fwd():
    w = workloads.make_random_vsa(2, 3, 64 * 9, 128, 64, 6, seed=62, vbs_lo=0, vbs_hi=64)
    out, lse = run_gpu(w)
    compare(w, out, lse)


@pytest.mark.parametrize("block", [64, 128])
def test_no_keys_gives_empty_rows(block):
    w = gqa(block, 63, Hq=4, Hkv=2, nbq=3, nbk=0, max_kv=2)
    out, lse = run_gpu(w)
    assert torch.equal(out, torch.zeros_like(out))
    assert bool((lse == binding.LSE_EMPTY).all())
    compare(w, out, lse)


@pytest.mark.parametrize("block", [64, 128])
def test_gqa_without_tail_masks_and_no_lse(block):
    w = gqa(block, 64, Hq=6, Hkv=3, nbq=5, nbk=7)
    dev = to_dev(w)
    out1, lse1 = binding.vsa_fwd_gqa(dev["q"], dev["k"], dev["v"], dev["idx"], dev["num"], None,
                                     block=block, scale=w.scale)
    out2, l2 = binding.vsa_fwd_gqa(dev["q"], dev["k"], dev["v"], dev["idx"], dev["num"], None,
                                   block=block, scale=w.scale, lse=False)
    torch.cuda.synchronize()
    assert l2 is None and torch.equal(out1, out2)
    w.vbs = np.full(w.nbk, block, np.int32)
    compare(w, out1, lse1)


# ------------------------------------------------------------------ from a block map
@pytest.mark.parametrize("block", [64, 128])
@pytest.mark.parametrize("shared", [False, True])
def test_from_mask(block, shared):
    w = gqa(block, 70 + shared, B=2, Hq=4, Hkv=2, nbq=7, nbk=9, kind="mask", shared_map=shared)
    out, lse = run_gpu(w)
    compare(w, out, lse)


@pytest.mark.parametrize("block", [64, 128])
def test_from_mask_equals_lut_of_the_same_map(block):
    # both routes hand the kernel the same ascending key-block list, so the results are
    # bit-identical
    w = gqa(block, 72, B=1, Hq=4, Hkv=1, nbq=6, nbk=11, kind="mask", max_kv=9)
    dev = to_dev(w)
    out_m, lse_m = binding.vsa_fwd_from_mask(dev["q"], dev["k"], dev["v"], dev["map"],
                                             dev["vbs"], block=block, scale=w.scale)
    idx, num = binding.vsa_bitmap_to_lut(dev["map"], w.nbk)
    out_l, lse_l = binding.vsa_fwd_gqa(dev["q"], dev["k"], dev["v"], idx, num, dev["vbs"],
                                       block=block, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(out_m, out_l) and torch.equal(lse_m, lse_l)


def test_from_mask_bool_map_and_dynamic_schedule():
    w = gqa(64, 73, B=1, Hq=2, Hkv=2, nbq=8, nbk=8, kind="mask")
    dev = to_dev(w)
    ref, ref_lse = run_gpu(w, dev)
    ws = binding.new_workspace()
    out, lse = binding.vsa_fwd_from_mask(dev["q"], dev["k"], dev["v"], dev["map"].bool(),
                                         dev["vbs"], block=64, scale=w.scale, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out, ref) and torch.equal(lse, ref_lse)
    assert int(ws.abs().sum()) == 0


# ------------------------------------------------------------- a larger grouped case
def test_large_gqa_sampled():
    # 16 query heads on 4 key/value heads, 16k queries over 24k keys, 64 of 384 blocks
    w = workloads.make_random_gqa(1, 16, 4, 16384, 24576, 128, 64, 64, seed=80, n_lo=64,
                                  n_hi=64, vbs_lo=48, vbs_hi=64)
    out, lse = run_gpu(w, workspace=binding.new_workspace())
    sel = sample_qblocks(w.B, w.H, w.nbq, 8, seed=1, must=(1,))
    compare(w, out, lse, sel)


# --------------------------------------------------- the largest key-block count accepted
@pytest.mark.parametrize("block", [64, 128])
@pytest.mark.parametrize("route", ["lut", "mask", "split"])
def test_max_key_blocks_every_block_selected(route, block):
    # 2048 key blocks (VSA_MAX_BLOCKS), every one selected by every query block: the
    # longest list the kernel builds, a dense row of 131,072 (block 64) or 262,144 keys
    nbk = binding.MAX_BLOCKS
    w = workloads.make_random_gqa(1, 2, 1, 128, nbk * block, 128, block, nbk, seed=150,
                                  n_lo=nbk, kind="mask" if route == "mask" else "vsa",
                                  vbs_lo=block - 4, vbs_hi=block)
    assert int(w.q2k_num.min()) == nbk
    out, lse = run_gpu(w, splits=8 if route == "split" else None)
    compare(w, out, lse)
