"""Randomised parity sweep: seeded random small configurations through the forward (LUT or
grouped-head route, every third case also split-KV) and the backward, and through the two
block-map routes (a shared Jenga bitmap, a per-head map for vsa_fwd_from_mask), each compared
with the oracle at the contract's tolerances (gpu_util for the forward; the backward bounds
of test_bwd_gpu.py).

A case draws the block size (64 or 128), 1-2 batches, 1-2 key/value heads with 1-3 query
heads each, 1-8 query blocks, 1-10 key blocks (so Sq and Sk differ, and a block-64 head can
have an odd number of query blocks), max_kv from 1 to nbk + 2, tail masks 0..block, and
occasionally peaky scores (q and k x3).  The LUT is then abused the way the contract
tolerates ("FastVideo block_sparse_attn_sm100a.py", `is_supported` docstring: padding is
never dereferenced; TheRock page: the block list is a set): -1 padding and out-of-range
entries below the count, duplicated entries, counts below 0 and above max_kv.  The oracle
reads the same LUT with its set / skip / clamp semantics.
"""
import numpy as np
import pytest
import torch

from block_sparse_attention_vsa_gb300 import binding, workloads
from oracle import oracle as orc
from gpu_util import compare, run_gpu, to_dev

pytestmark = pytest.mark.gpu

N_CASES = 48
BWD_REL_MAX, BWD_REL_MEAN = 2e-2, 1.5e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def random_case(seed):
    rng = np.random.default_rng(7000 + seed)
    block = int(rng.choice([64, 128]))
    B = int(rng.integers(1, 3))
    Hkv = int(rng.integers(1, 3))
    group = int(rng.integers(1, 4))
    nbq = int(rng.integers(1, 9))
    nbk = int(rng.integers(1, 11))
    max_kv = int(rng.integers(1, nbk + 3))
    qk_mul = 3.0 if rng.random() < 0.25 else 1.0
    w = workloads.make_random_gqa(B, Hkv * group, Hkv, nbq * block, nbk * block, 128, block,
                                  max_kv, seed=9000 + seed, vbs_lo=0, vbs_hi=block,
                                  qk_mul=qk_mul)
    idx = w.q2k_idx
    num = w.q2k_num
    u = rng.random(idx.shape)
    idx[u < 0.06] = -1                          # padding below the count
    idx[(u >= 0.06) & (u < 0.10)] = nbk + 5     # out of range below the count
    if max_kv >= 2:                             # duplicates: slot 1 repeats slot 0
        d = rng.random(idx.shape[:3]) < 0.2
        idx[..., 1][d] = idx[..., 0][d]
    c = rng.random(num.shape)
    num[c < 0.05] = -3                          # negative count: nothing selected
    num[(c >= 0.05) & (c < 0.10)] = max_kv + 4  # count above max_kv: clamped
    return w


def backward_compare(w, dev, out, lse, seed):
    g = torch.Generator().manual_seed(seed)
    do = torch.randn(w.q.shape, generator=g).to(torch.bfloat16)
    dq, dk, dv = binding.vsa_bwd(dev["q"], dev["k"], dev["v"], out, do.to(dev["q"].device), lse,
                                 dev["idx"], dev["num"], dev["vbs"], block=w.block,
                                 scale=w.scale)
    torch.cuda.synchronize()
    code, detail = binding.vsa_device_status()
    assert code == binding.VSA_OK, hex(detail)
    refs = orc.vsa_backward(workloads.bits(w.q), workloads.bits(w.k), workloads.bits(w.v),
                            workloads.bits(do), w.q2k_idx, w.q2k_num, w.vbs, w.block, w.scale)
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        got = got.float().cpu().numpy().astype(np.float64)
        scale_max, scale_mean = np.abs(ref).max(), np.abs(ref).mean()
        if scale_max == 0.0:
            assert np.all(got == 0.0), name
            continue
        e = np.abs(got - ref)
        assert e.max() <= BWD_REL_MAX * scale_max, (name, e.max(), scale_max)
        assert e.mean() <= BWD_REL_MEAN * scale_mean, (name, e.mean(), scale_mean)


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_case(seed):
    w = random_case(seed)
    dev = to_dev(w)
    out, lse = run_gpu(w, dev)
    compare(w, out, lse)
    if seed % 3 == 0:
        splits = 2 + seed % 4
        # the workspace's schedule counters start at zero (the library's allocator)
        ws = binding.new_split_workspace(w.B, w.H, w.S, w.block, splits)
        out_s, lse_s = run_gpu(w, dev, workspace=ws, splits=splits)
        compare(w, out_s, lse_s)
    backward_compare(w, dev, out, lse, seed)


def random_mask_case(seed):
    """A block-map case: even seeds a Jenga map shared by every head (square, no grouping, no
    tail masks), odd seeds a per-head int8 map for vsa_fwd_from_mask (grouped heads, cross
    length, tail masks).  Density is drawn per case; selected bytes take any nonzero value."""
    rng = np.random.default_rng(8000 + seed)
    block = int(rng.choice([64, 128]))
    B = int(rng.integers(1, 3))
    jenga = seed % 2 == 0
    if jenga:
        Hkv = Hq = int(rng.integers(1, 4))
        nbq = nbk = int(rng.integers(1, 10))
    else:
        Hkv = int(rng.integers(1, 3))
        Hq = Hkv * int(rng.integers(1, 4))
        nbq, nbk = int(rng.integers(1, 9)), int(rng.integers(1, 11))
    qk_mul = 3.0 if rng.random() < 0.25 else 1.0
    w = workloads.make_random_gqa(B, Hq, Hkv, nbq * block, nbk * block, 128, block, nbk,
                                  seed=9500 + seed, vbs_lo=None if jenga else 0,
                                  vbs_hi=None if jenga else block, kind="mask",
                                  shared_map=jenga, qk_mul=qk_mul)
    shape = (nbq, nbk) if jenga else (B, Hq, nbq, nbk)
    values = rng.integers(-128, 128, size=shape).astype(np.int8)
    values[values == 0] = 1
    bm = np.where(rng.random(shape) < rng.uniform(0.0, 1.0), values, 0).astype(np.int8)
    if jenga:
        return workloads.Workload(name="jenga_random", kind="jenga", B=B, H=Hq, S=w.S, D=w.D,
                                  block=block, scale=w.scale, q=w.q, k=w.k, v=w.v,
                                  bitmap=np.ascontiguousarray(bm))
    w.block_map = np.ascontiguousarray(bm)
    return w


@pytest.mark.parametrize("seed", range(16))
def test_random_mask_case(seed):
    w = random_mask_case(seed)
    out, lse = run_gpu(w, to_dev(w))
    compare(w, out, lse)
