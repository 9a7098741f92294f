"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the same seeded
inputs, element by element, with the contract's tolerances (tests/gpu_util.py).

Small cases (every row) span several key tiles, odd unions (a ragged N = 64 last tile),
ragged counts and tail masks; the full-size workloads are checked on every row (tiny,
mid) or on a seeded sample of >= 16 query blocks per head that always includes the
first and last block (which carries the long-video tail mask).
"""
import numpy as np
import pytest
import torch

from block_sparse_attention_vsa_gb300 import binding, workloads
from oracle import oracle as orc
from gpu_util import compare, run_gpu, sample_qblocks, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def small(block, seed, B=2, H=3, nbk=16, max_kv=7, n_lo=0, n_hi=None, vbs=True, qk_mul=1.0):
    return workloads.make_random_vsa(B, H, nbk * block, 128, block, max_kv, seed, n_lo=n_lo,
                                     n_hi=n_hi, vbs_lo=0 if vbs else None,
                                     vbs_hi=block if vbs else None, qk_mul=qk_mul)


# ------------------------------------------------------------------------- small cases
def test_tiny_workload_every_row():
    w = workloads.make_vsa_tiny()
    out, lse = run_gpu(w)
    compare(w, out, lse)


@pytest.mark.parametrize("block", [64, 128])
@pytest.mark.parametrize("seed", [1, 2, 3])
def test_random_ragged(block, seed):
    w = small(block, seed)
    out, lse = run_gpu(w)
    compare(w, out, lse)


@pytest.mark.parametrize("block", [64, 128])
@pytest.mark.parametrize("mul", [4.0, 8.0])
def test_peaky_softmax_rescales(block, mul):
    # q, k x 8: scores of std ~90 in log2 units, so the running max jumps by more than the
    # 2^32 lag allowed before a rescale of O and l many times per row
    w = small(block, 11, max_kv=12, n_lo=6, qk_mul=mul)
    out, lse = run_gpu(w)
    compare(w, out, lse)


@pytest.mark.parametrize("block", [64, 128])
def test_large_values_under_a_lagging_max(block):
    # V x 2^10 (exact in bf16) on peaky scores: P up to 2^32 times V up to ~2^12 summed
    # over 24 key blocks must stay finite, and out must be exactly 2^10 times the
    # oracle's out for the unscaled V within the tolerance scaled by 2^10
    w = small(block, 12, max_kv=24, n_lo=16, qk_mul=3.0)
    dev = to_dev(w)
    dev["v"] = dev["v"] * 1024.0
    out, lse = run_gpu(w, dev)
    assert bool(torch.isfinite(out.float()).all()) and bool(torch.isfinite(lse).all())
    compare(w, (out.float() / 1024.0).to(torch.bfloat16), lse)


@pytest.mark.parametrize("block", [64, 128])
def test_dense_all_blocks(block):
    nbk = 8
    w = small(block, 5, B=1, H=2, nbk=nbk, max_kv=nbk, vbs=False)
    w.q2k_idx[:] = np.arange(nbk, dtype=np.int32)
    w.q2k_num[:] = nbk
    out, lse = run_gpu(w)
    compare(w, out, lse)


@pytest.mark.parametrize("block", [64, 128])
def test_all_rows_empty(block):
    w = small(block, 6)
    w.q2k_num[:] = 0
    out, lse = run_gpu(w)
    assert torch.all(out == 0) and not torch.any(torch.signbit(out.float()))
    assert torch.all(lse == binding.LSE_EMPTY)
    compare(w, out, lse)


@pytest.mark.parametrize("block", [64, 128])
def test_tail_mask_edges(block):
    w = small(block, 7, max_kv=10, n_lo=4)
    edge = np.array([0, 1, block - 1, block], np.int32)
    w.vbs[:] = edge[np.arange(w.nb) % 4]
    out, lse = run_gpu(w)
    compare(w, out, lse)


@pytest.mark.parametrize("block", [64, 128])
def test_selected_blocks_all_zero_width(block):
    # rows whose every selected block has no valid key are empty rows too
    w = small(block, 8, max_kv=5, n_lo=1)
    w.vbs[:] = 0
    w.vbs[1] = block
    out, lse = run_gpu(w)
    compare(w, out, lse)


@pytest.mark.parametrize("block", [64, 128])
def test_padding_never_read(block):
    w = small(block, 9)
    dev = to_dev(w)
    ref_out, ref_lse = run_gpu(w, dev)
    poisoned = w.q2k_idx.copy()
    slot = np.arange(w.max_kv)[None, None, None, :]
    pad = slot >= w.q2k_num[..., None]
    rng = np.random.default_rng(0)
    poisoned[pad] = rng.choice([2 ** 30, -2 ** 30, 0, w.nb - 1], size=int(pad.sum()))
    dev["idx"] = torch.from_numpy(poisoned).cuda()
    out, lse = run_gpu(w, dev)
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


@pytest.mark.parametrize("block", [64, 128])
def test_out_of_range_entries_and_clamped_counts(block):
    w = small(block, 10, max_kv=6, n_lo=3)
    rng = np.random.default_rng(1)
    w.q2k_idx[rng.random(w.q2k_idx.shape) < 0.2] = -3
    w.q2k_idx[rng.random(w.q2k_idx.shape) < 0.1] = w.nb + 5
    w.q2k_num[rng.random(w.q2k_num.shape) < 0.2] = 100   # clamped to max_kv
    w.q2k_num[rng.random(w.q2k_num.shape) < 0.1] = -7    # clamped to 0
    out, lse = run_gpu(w)
    compare(w, out, lse)


@pytest.mark.parametrize("block", [64, 128])
def test_duplicate_entries_attend_once(block):
    w = small(block, 12, max_kv=8, n_lo=4)
    w.q2k_idx[..., 1] = w.q2k_idx[..., 0]
    w.q2k_idx[..., 3] = w.q2k_idx[..., 0]
    out, lse = run_gpu(w)
    compare(w, out, lse)


@pytest.mark.parametrize("block", [64, 128])
def test_slot_order_does_not_matter(block):
    w = small(block, 13, max_kv=8, n_lo=8)
    ref_out, ref_lse = run_gpu(w)
    rng = np.random.default_rng(2)
    w.q2k_idx = np.ascontiguousarray(w.q2k_idx[..., rng.permutation(w.max_kv)])
    out, lse = run_gpu(w)
    # the kernel walks selected blocks in ascending order whatever the slot order
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


@pytest.mark.parametrize("block", [64, 128])
def test_jenga_small(block):
    B, H, nbk = 1, 3, 16
    g = workloads.gen(21)
    q, k, v = workloads.make_qkv(B, H, nbk * block, 128, g, mul_qk=3.0)
    bm = workloads.jenga_bitmap(nbk, g, lo=-2, hi=1, extra=2)
    bm[3, :] = 0                       # one empty query block
    bm[5, 7] = 57                      # any nonzero byte means attend
    w = workloads.Workload("jenga_small", "jenga", B, H, nbk * block, 128, block, 128 ** -0.5,
                           q, k, v, bitmap=bm)
    out, lse = run_gpu(w)
    compare(w, out, lse)


@pytest.mark.parametrize("block", [64, 128])
def test_no_lse_route_same_output(block):
    w = small(block, 14)
    dev = to_dev(w)
    out1, _ = run_gpu(w, dev)
    out2, l2 = run_gpu(w, dev, lse=False)
    assert l2 is None and torch.equal(out1, out2)


@pytest.mark.parametrize("block", [64, 128])
def test_dynamic_schedule_matches_static(block):
    w = small(block, 15)
    dev = to_dev(w)
    ws = binding.new_workspace()
    out_s, lse_s = run_gpu(w, dev)
    for _ in range(2):
        out_d, lse_d = run_gpu(w, dev, workspace=ws)
        assert torch.equal(out_s, out_d) and torch.equal(lse_s, lse_d)
        assert int(ws.abs().sum()) == 0, "workspace not returned to zero"


def test_int64_metadata_is_cast():
    w = small(64, 16)
    dev = to_dev(w)
    ref_out, ref_lse = run_gpu(w, dev)
    out, lse = binding.vsa_fwd(dev["q"], dev["k"], dev["v"], dev["idx"].long(), dev["num"].long(),
                               dev["vbs"].long(), scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


def test_from_host_buffers():
    w = small(64, 17)
    dev = to_dev(w)
    ref_out, ref_lse = run_gpu(w, dev)
    h = dict(q=w.q.pin_memory(), k=w.k.pin_memory(), v=w.v.pin_memory(),
             idx=torch.from_numpy(w.q2k_idx).pin_memory(),
             num=torch.from_numpy(w.q2k_num).pin_memory(),
             vbs=torch.from_numpy(w.vbs).pin_memory())
    h_out = torch.empty_like(w.q).pin_memory()
    h_lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32).pin_memory()
    bufs = {kk: torch.empty_like(t) for kk, t in dev.items()}
    bufs["out"] = torch.empty_like(dev["q"])
    bufs["lse"] = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device="cuda")
    binding.vsa_fwd_from_host(h["q"], h["k"], h["v"], h["idx"], h["num"], h["vbs"], w.block,
                              w.scale, h_out, h_lse, bufs)
    torch.cuda.synchronize()
    assert torch.equal(h_out, ref_out.cpu()) and torch.equal(h_lse, ref_lse.cpu())


def host_chunks(B, H, S):
    """Chunks vsa_fwd_from_host makes: about 20 MB of q, k, v each, at most 32, at most one
    per (b, h) head."""
    n = -(-(B * H * 3 * S * 128 * 2) // (20 << 20))
    return min(max(1, min(32, n)), B * H)


@pytest.mark.parametrize("block,B,H,nbk,with_lse,dynamic", [(64, 2, 5, 16, True, False),
                                                              (128, 1, 3, 16, False, True),
                                                              (64, 1, 11, 128, True, True),
                                                              (128, 2, 7, 64, True, False)])
def test_from_host_chunks_on_a_side_stream(block, B, H, nbk, with_lse, dynamic):
    """The host-buffer entry splits the heads into chunks (uneven ones included: the two
    larger cases make 4 and 5 chunks of 11 and 14 heads) whose copies overlap other chunks'
    forwards on internal streams forked from the caller's stream; the result equals
    vsa_fwd's bit for bit (and, on the small cases, the oracle's within tolerance), and work
    enqueued on the caller's stream afterwards sees the copies complete."""
    w = small(block, 23 + H, B=B, H=H, nbk=nbk)
    dev = to_dev(w)
    ref_out, ref_lse = run_gpu(w, dev)
    if nbk <= 16:
        compare(w, ref_out, ref_lse)
    h = dict(q=w.q.pin_memory(), k=w.k.pin_memory(), v=w.v.pin_memory(),
             idx=torch.from_numpy(w.q2k_idx).pin_memory(),
             num=torch.from_numpy(w.q2k_num).pin_memory(),
             vbs=torch.from_numpy(w.vbs).pin_memory())
    h_out = torch.full_like(w.q, float("nan")).pin_memory()
    h_lse = torch.full((w.B, w.H, w.S), float("nan"), dtype=torch.float32).pin_memory()
    bufs = {kk: torch.zeros_like(t) for kk, t in dev.items()}
    bufs["out"] = torch.empty_like(dev["q"])
    bufs["lse"] = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    ws = binding.new_workspace(dev["q"].device) if dynamic else None
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        binding.vsa_fwd_from_host(h["q"], h["k"], h["v"], h["idx"], h["num"], h["vbs"], w.block,
                                  w.scale, h_out, h_lse if with_lse else None, bufs,
                                  workspace=ws, stream=side)
        # enqueued after the call on the same stream: must see every chunk's copy done
        probe = bufs["out"].float().sum()
    side.synchronize()
    assert binding.vsa_last_launch_count() == host_chunks(B, H, w.S)
    assert torch.equal(h_out, ref_out.cpu())
    assert torch.equal(bufs["q"], dev["q"]) and torch.equal(bufs["idx"], dev["idx"])
    assert probe.item() == ref_out.float().sum().item()
    if with_lse:
        assert torch.equal(h_lse, ref_lse.cpu())
    code, detail = binding.vsa_device_status()
    assert code == binding.VSA_OK, hex(detail)


def test_host_chunk_counts():
    """The chunk rule on the benchmark shapes: one-head chunks for B1 H24 S98304, eight for
    B1 H12 S16384, the cap of 32 for B2 H24 S32768."""
    assert host_chunks(1, 24, 98304) == 24
    assert host_chunks(1, 12, 16384) == 8
    assert host_chunks(2, 24, 32768) == 32
    assert host_chunks(1, 11, 8192) == 4 and host_chunks(2, 7, 8192) == 5


# ------------------------------------------------------------- metadata conversions
def test_lut_to_bitmap_bit_exact():
    rng = np.random.default_rng(3)
    rows, max_kv, nb = 300, 9, 40
    idx = rng.integers(-4, nb + 4, size=(rows, max_kv)).astype(np.int32)
    num = rng.integers(-2, max_kv + 4, size=rows).astype(np.int32)
    got = binding.vsa_lut_to_bitmap(torch.from_numpy(idx).cuda(), torch.from_numpy(num).cuda(), nb)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), orc.lut_to_blockmask(idx, num, nb))


@pytest.mark.parametrize("max_kv", [1, 5, 40, 77])
def test_bitmap_to_lut_bit_exact(max_kv):
    rng = np.random.default_rng(4)
    rows, nb = 257, 70
    bm = (rng.random((rows, nb)) < 0.3).astype(np.int8) * rng.integers(1, 100, size=(rows, nb)).astype(np.int8)
    bm[0] = 0
    bm[1] = 1
    gi, gn = binding.vsa_bitmap_to_lut(torch.from_numpy(bm).cuda(), max_kv)
    torch.cuda.synchronize()
    ri, rn = orc.blockmask_to_lut(bm, max_kv)
    assert np.array_equal(gi.cpu().numpy(), ri) and np.array_equal(gn.cpu().numpy(), rn)


def test_device_conversions_round_trip_on_workload():
    w = workloads.make_vsa_tiny()
    idx, num = torch.from_numpy(w.q2k_idx).cuda(), torch.from_numpy(w.q2k_num).cuda()
    bm = binding.vsa_lut_to_bitmap(idx, num, w.nb)
    i2, n2 = binding.vsa_bitmap_to_lut(bm, w.max_kv)
    torch.cuda.synchronize()
    ri, rn = orc.blockmask_to_lut(orc.lut_to_blockmask(w.q2k_idx, w.q2k_num, w.nb), w.max_kv)
    assert np.array_equal(i2.cpu().numpy(), ri) and np.array_equal(n2.cpu().numpy(), rn)


# ------------------------------------------------------------------ full-size workloads
def test_mid_workload_every_row():
    w = workloads.make("vsa_mid")
    out, lse = run_gpu(w)
    compare(w, out, lse)


@pytest.mark.parametrize("name", ["vsa_blk128", "jenga", "vsa_long_video"])
def test_full_workload_sampled(name):
    w = workloads.make(name)
    out, lse = run_gpu(w, workspace=binding.new_workspace())
    sel = sample_qblocks(w.B, w.H, w.nb, 16, seed=0, must=(1, w.nb // 2))
    compare(w, out, lse, sel)


def test_launch_count_and_status():
    w = small(64, 18)
    run_gpu(w)
    assert binding.vsa_last_launch_count() == 1
    code, detail = binding.vsa_device_status()
    assert code == binding.VSA_OK and detail == 0
