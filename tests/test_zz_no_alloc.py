"""vsa_fwd_noalloc: the forward for callers that cannot give the library device memory of
their own (a plug-in whose host framework owns every allocation, or a serving loop that
must not call cudaMalloc once running).  Its scheduling scratch is a static array inside
the library.  This test calls it through the C ABI twice in a row and checks both
results against vsa_fwd (which takes a caller workspace).  Both run the same kernel with
the same dynamic schedule, and every work item's arithmetic is independent of which CTA
claims it, so the outputs must be bit-identical; vsa_fwd itself is also held to the oracle
at the parity tolerances of the other GPU tests.  The file is named to be collected last.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from block_sparse_attention_vsa_gb300 import binding
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return binding.load()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("block", [64, 128])
def test_noalloc_matches_vsa_fwd_twice(lib, block):
    from block_sparse_attention_vsa_gb300 import binding, workloads
    w = workloads.make_random_vsa(2, 3, 16 * block, 128, block, 7, seed=31, n_lo=0,
                                  vbs_lo=0, vbs_hi=block)
    d = torch.device("cuda:0")
    q, k, v = (t.to(d) for t in (w.q, w.k, w.v))
    idx, num, vbs = (torch.from_numpy(x).to(d) for x in (w.q2k_idx, w.q2k_num, w.vbs))
    ref_out, ref_lse = binding.vsa_fwd(q, k, v, idx, num, vbs, block=block, scale=w.scale,
                                       workspace=binding.new_workspace(d))
    torch.cuda.synchronize()
    import gpu_util
    gpu_util.compare(w, ref_out, ref_lse)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        lse = torch.full((w.B, w.H, w.S), float("nan"), dtype=torch.float32, device=d)
        code = lib.vsa_fwd_noalloc(_p(q), _p(k), _p(v), _p(idx), _p(num), _p(vbs), w.B, w.H, w.S,
                                   w.D, w.max_kv, block, w.scale, _p(out), _p(lse), stream)
        assert code == binding.VSA_OK, lib.vsa_status_str(code)
        torch.cuda.synchronize()
        status, detail = binding.vsa_device_status()
        assert status == binding.VSA_OK, hex(detail)
        assert torch.equal(out, ref_out)
        assert torch.equal(lse, ref_lse)


def test_noalloc_rejects_what_vsa_fwd_rejects(lib):
    from block_sparse_attention_vsa_gb300 import binding
    P = ctypes.c_void_p
    # head dim 64 is not built: rejected before anything is enqueued
    code = lib.vsa_fwd_noalloc(P(1 << 20), P(2 << 20), P(3 << 20), P(4 << 20), P(5 << 20),
                               P(6 << 20), 1, 1, 256, 64, 4, 64, 0.1, P(7 << 20), None, None)
    assert code == binding.VSA_ERR_UNSUPPORTED
