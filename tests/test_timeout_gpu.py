"""Failure detection without a GPU fault.

Every internal wait of the forward and backward kernels is bounded.  A wait that runs out
records a code in the device status word, raises the CTA's abort flag, and every role of
the CTA returns after draining the copies and MMAs it has in flight; the host reads
VSA_ERR_DEVICE_TIMEOUT from vsa_device_status() and the context stays usable.  These
tests make waits run out on purpose, through the library's two test hooks (no trap, no
bad address, no endless loop):
  - the stall hook: the MMA warp waits on a barrier that nothing completes;
  - a 1 ns limit on every non-drain wait, so ordinary waits give up mid-pipeline while
    copies and MMAs are in flight (drain waits keep their full limit).
After each, an ordinary call on the same context must match the oracle.
"""
import numpy as np
import pytest
import torch

import gpu_util

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from block_sparse_attention_vsa_gb300 import binding
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return binding.load()


@pytest.fixture
def hooks(lib):
    from block_sparse_attention_vsa_gb300 import binding
    yield binding
    binding.vsa_set_stall_test(False)
    binding.vsa_set_wait_limit_ns(0)


def _launch_fwd(binding, w, dev, workspace=None):
    if w.kind == "vsa":
        return binding.vsa_fwd(dev["q"], dev["k"], dev["v"], dev["idx"], dev["num"], dev["vbs"],
                               block=w.block, scale=w.scale, workspace=workspace)
    return binding.jenga_fwd(dev["q"], dev["k"], dev["v"], dev["bitmap"], w.block, w.block,
                             scale=w.scale, workspace=workspace)


def _recovers(w, dev):
    """An ordinary call on the same context matches the oracle and leaves status OK."""
    out, lse = gpu_util.run_gpu(w, dev)
    gpu_util.compare(w, out, lse)


@pytest.mark.parametrize("block,dynamic", [(64, False), (128, True)])
def test_forward_stall_reports_timeout(hooks, block, dynamic):
    from block_sparse_attention_vsa_gb300 import workloads
    binding = hooks
    w = workloads.make_random_vsa(1, 4, 16 * block, 128, block, 8, seed=41, n_lo=1)
    dev = gpu_util.to_dev(w)
    ws = binding.new_workspace(dev["q"].device) if dynamic else None
    binding.vsa_set_wait_limit_ns(10_000_000)  # 10 ms instead of about a second
    binding.vsa_set_stall_test(True)
    _launch_fwd(binding, w, dev, ws)
    torch.cuda.synchronize()
    code, detail = binding.vsa_device_status()
    binding.vsa_set_stall_test(False)
    binding.vsa_set_wait_limit_ns(0)
    assert code == binding.VSA_ERR_DEVICE_TIMEOUT, (code, hex(detail))
    assert detail & 0xF00 == 0x100, hex(detail)
    # the dynamic schedule's counters must be back at zero for the next call to use
    if ws is not None:
        assert int(ws.abs().sum().item()) == 0
    out, lse = gpu_util.run_gpu(w, dev, workspace=ws)
    gpu_util.compare(w, out, lse)


def test_jenga_stall_reports_timeout(hooks):
    from block_sparse_attention_vsa_gb300 import workloads
    binding = hooks
    w = workloads.make_random_vsa(1, 2, 24 * 64, 128, 64, 8, seed=43, n_lo=1)
    # the same selection as a block map shared by both heads: head 0's rows
    from oracle import oracle as orc
    bitmap = orc.lut_to_blockmask(w.q2k_idx[:, :1], w.q2k_num[:, :1], w.nbk)[0, 0]
    jw = workloads.Workload(name="jenga_small", kind="jenga", B=w.B, H=w.H, S=w.S, D=w.D,
                            block=w.block, scale=w.scale, q=w.q, k=w.k, v=w.v,
                            bitmap=np.ascontiguousarray(bitmap.astype(np.int8)))
    dev = gpu_util.to_dev(jw)
    binding.vsa_set_wait_limit_ns(10_000_000)
    binding.vsa_set_stall_test(True)
    _launch_fwd(binding, jw, dev)
    torch.cuda.synchronize()
    code, detail = binding.vsa_device_status()
    binding.vsa_set_stall_test(False)
    binding.vsa_set_wait_limit_ns(0)
    assert code == binding.VSA_ERR_DEVICE_TIMEOUT, (code, hex(detail))
    _recovers(jw, dev)


def test_forward_short_limit_gives_up_mid_pipeline(hooks):
    """A 1 ns limit on the non-drain waits: waits give up while copies and MMAs are in
    flight.  Several launches must report the timeout between them (a single launch can
    in principle see every phase complete on the first poll), each is followed by a clean
    call."""
    from block_sparse_attention_vsa_gb300 import workloads
    binding = hooks
    timeouts = 0
    for seed, block in ((51, 64), (52, 128), (53, 64)):
        w = workloads.make_random_vsa(1, 8, 32 * block, 128, block, 16, seed=seed, n_lo=4)
        dev = gpu_util.to_dev(w)
        binding.vsa_set_wait_limit_ns(1)
        _launch_fwd(binding, w, dev)
        torch.cuda.synchronize()
        code, detail = binding.vsa_device_status()
        binding.vsa_set_wait_limit_ns(0)
        assert code in (binding.VSA_OK, binding.VSA_ERR_DEVICE_TIMEOUT), code
        if code == binding.VSA_ERR_DEVICE_TIMEOUT:
            assert detail & 0xF00 == 0x100, hex(detail)
            timeouts += 1
        _recovers(w, dev)
    assert timeouts >= 1


@pytest.mark.parametrize("block", [64, 128])
def test_backward_stall_reports_timeout(hooks, block):
    """The backward kernel unwinds from a stalled MMA warp, on 128-key blocks and on
    pairs of 64-key blocks."""
    from block_sparse_attention_vsa_gb300 import workloads
    binding = hooks
    w = workloads.make_random_vsa(1, 2, 8 * block, 128, block, 4, seed=47, n_lo=1)
    dev = gpu_util.to_dev(w)
    out, lse = binding.vsa_fwd(dev["q"], dev["k"], dev["v"], dev["idx"], dev["num"], dev["vbs"],
                               block=w.block, scale=w.scale)
    g = torch.Generator().manual_seed(2)
    dout_cpu = torch.randn(w.q.shape, generator=g).to(torch.bfloat16)
    dout = dout_cpu.to(dev["q"].device)
    binding.vsa_set_wait_limit_ns(10_000_000)
    binding.vsa_set_stall_test(True)
    binding.vsa_bwd(dev["q"], dev["k"], dev["v"], out, dout, lse, dev["idx"], dev["num"],
                    dev["vbs"], block=w.block, scale=w.scale)
    torch.cuda.synchronize()
    code, detail = binding.vsa_device_status()
    binding.vsa_set_stall_test(False)
    binding.vsa_set_wait_limit_ns(0)
    assert code == binding.VSA_ERR_DEVICE_TIMEOUT, (code, hex(detail))
    assert detail & 0xF00 == 0x100, hex(detail)
    # the same backward again, now clean, against the oracle
    dq, dk, dv = binding.vsa_bwd(dev["q"], dev["k"], dev["v"], out, dout, lse, dev["idx"],
                                 dev["num"], dev["vbs"], block=w.block, scale=w.scale)
    torch.cuda.synchronize()
    code, detail = binding.vsa_device_status()
    assert code == binding.VSA_OK, hex(detail)
    from oracle import oracle as orc
    refs = orc.vsa_backward(workloads.bits(w.q), workloads.bits(w.k), workloads.bits(w.v),
                            workloads.bits(dout_cpu), w.q2k_idx, w.q2k_num, w.vbs, w.block, w.scale)
    for got, ref in zip((dq, dk, dv), refs):
        e = np.abs(got.float().cpu().numpy().astype(np.float64) - ref)
        assert e.max() <= 2e-2 * np.abs(ref).max()


@pytest.mark.parametrize("block", [64, 128])
def test_backward_short_limit_gives_up_mid_pipeline(hooks, block):
    """A 1 ns limit on the backward's non-drain waits: they give up while copies and MMAs
    are in flight (the drains keep their full limit).  At least one of the launches must
    report the timeout, and each is followed by a clean backward that matches the oracle."""
    from block_sparse_attention_vsa_gb300 import workloads
    from oracle import oracle as orc
    binding = hooks
    timeouts = 0
    for seed in (61, 62, 63):
        w = workloads.make_random_vsa(1, 4, 16 * block, 128, block, 8, seed=seed, n_lo=2)
        dev = gpu_util.to_dev(w)
        out, lse = binding.vsa_fwd(dev["q"], dev["k"], dev["v"], dev["idx"], dev["num"],
                                   dev["vbs"], block=w.block, scale=w.scale)
        g = torch.Generator().manual_seed(seed)
        dout_cpu = torch.randn(w.q.shape, generator=g).to(torch.bfloat16)
        dout = dout_cpu.to(dev["q"].device)
        binding.vsa_set_wait_limit_ns(1)
        binding.vsa_bwd(dev["q"], dev["k"], dev["v"], out, dout, lse, dev["idx"], dev["num"],
                        dev["vbs"], block=w.block, scale=w.scale)
        torch.cuda.synchronize()
        code, detail = binding.vsa_device_status()
        binding.vsa_set_wait_limit_ns(0)
        assert code in (binding.VSA_OK, binding.VSA_ERR_DEVICE_TIMEOUT), code
        if code == binding.VSA_ERR_DEVICE_TIMEOUT:
            assert detail & 0xF00 == 0x100, hex(detail)
            timeouts += 1
        dq, dk, dv = binding.vsa_bwd(dev["q"], dev["k"], dev["v"], out, dout, lse, dev["idx"],
                                     dev["num"], dev["vbs"], block=w.block, scale=w.scale)
        torch.cuda.synchronize()
        code, detail = binding.vsa_device_status()
        assert code == binding.VSA_OK, hex(detail)
        refs = orc.vsa_backward(workloads.bits(w.q), workloads.bits(w.k), workloads.bits(w.v),
                                workloads.bits(dout_cpu), w.q2k_idx, w.q2k_num, w.vbs, w.block,
                                w.scale)
        for got, ref in zip((dq, dk, dv), refs):
            e = np.abs(got.float().cpu().numpy().astype(np.float64) - ref)
            assert e.max() <= 2e-2 * np.abs(ref).max()
    assert timeouts >= 1
