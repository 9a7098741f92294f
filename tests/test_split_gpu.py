"""GPU parity for the split-KV forward (vsa_fwd_split): each work item's key tiles are cut
into num_splits ranges whose fp32 partials a second kernel merges.  Checked against the
fp64 oracle on the same seeded inputs (tolerances in tests/gpu_util.py), including more
ranges than tiles (empty ranges), odd query-block counts, tail masks, empty rows, grouped
heads and the full-size decode workload (a short query over a long context).

The merge follows the split-K pattern of "vLLM FlyDSL tq_decode" (a partial (m, l, O) per
key partition, then a reduction); the arithmetic of each range is that of vsa_fwd.
"""
import numpy as np
import pytest
import torch

from block_sparse_attention_vsa_gb300 import binding, workloads
from gpu_util import compare, run_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def case(block, seed, B=1, Hq=4, Hkv=2, nbq=2, nbk=40, max_kv=24, n_lo=0, **kw):
    return workloads.make_random_gqa(B, Hq, Hkv, nbq * block, nbk * block, 128, block, max_kv,
                                     seed, n_lo=n_lo, vbs_lo=0, vbs_hi=block, **kw)


@pytest.mark.parametrize("block", [64, 128])
@pytest.mark.parametrize("splits", [1, 2, 3, 7, 32])
def test_split_matches_oracle(block, splits):
    # 32 ranges for at most 24 tiles: some ranges are empty
    w = case(block, 90 + splits, n_lo=10)
    ws = binding.new_split_workspace(w.B, w.H, w.S, w.block, splits)
    out, lse = run_gpu(w, workspace=ws, splits=splits)
    compare(w, out, lse)
    assert int(ws[:64].abs().sum()) == 0, "scheduling counters not returned to zero"


@pytest.mark.parametrize("block", [64, 128])
def test_split_odd_blocks_empty_rows_and_no_lse(block):
    w = case(block, 95, B=2, Hq=3, Hkv=1, nbq=5, nbk=13, max_kv=9)
    w.q2k_num[0, 1, :] = 0  # a head with no attended key at all
    dev = to_dev(w)
    out, lse = run_gpu(w, dev, splits=4)
    compare(w, out, lse)
    out2, l2 = run_gpu(w, dev, lse=False, splits=4)
    assert l2 is None and torch.equal(out, out2)


def test_split_close_to_single_pass():
    w = case(64, 96, B=1, Hq=8, Hkv=8, nbq=4, nbk=64, max_kv=48, n_lo=40)
    dev = to_dev(w)
    ref, ref_lse = run_gpu(w, dev)
    out, lse = run_gpu(w, dev, splits=5)
    assert (out.float() - ref.float()).abs().max().item() <= 2e-2
    assert (lse - ref_lse).abs().max().item() <= 1e-3
    assert binding.vsa_last_launch_count() == 2


def test_split_rejects_a_small_workspace():
    w = case(64, 97)
    dev = to_dev(w)
    need = binding.split_workspace_bytes(w.B, w.H, w.S, w.block, 3)
    small = torch.zeros((need - 256) // 4, dtype=torch.int32, device="cuda")
    with pytest.raises(binding.VsaError) as e:
        run_gpu(w, dev, workspace=small, splits=3)
    assert e.value.code == binding.VSA_ERR_INVALID_ARG


def test_decode_workload_every_row():
    w = workloads.make("vsa_decode")
    n = binding.default_splits(w.B, w.H, w.S, w.block,
                               torch.cuda.get_device_properties(0).multi_processor_count)
    assert n > 1
    out, lse = run_gpu(w, splits=n)
    compare(w, out, lse)
