"""The C-ABI library loads and exports every entry point include/vsa.h declares; host-side
argument checks reject bad calls with the documented status before touching the GPU.
Runs without a GPU (no compute calls)."""
import ctypes
import os
import re

import pytest

from block_sparse_attention_vsa_gb300 import binding
from block_sparse_attention_vsa_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vsa.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vsa_\w+|jenga_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return binding.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("vsa_fwd", "jenga_fwd", "vsa_lut_to_bitmap", "vsa_bitmap_to_lut"):
        assert n in names
    assert set(names) == set(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_library_has_sm103a_code_only():
    # the build passes exactly one -gencode, for sm_103a
    assert libbuild.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_status_strings(lib):
    for code in range(5):
        assert lib.vsa_status_str(code)


NULL = None


def _fwd(lib, **kw):
    args = dict(q=1 << 20, k=2 << 20, v=3 << 20, idx=4 << 20, num=5 << 20, vbs=6 << 20, B=1, H=1,
                S=256, D=128, max_kv=4, block=64, scale=0.088, out=7 << 20, lse=None, ws=None)
    args.update(kw)
    P = ctypes.c_void_p
    return lib.vsa_fwd(P(args["q"]), P(args["k"]), P(args["v"]), P(args["idx"]), P(args["num"]),
                       P(args["vbs"]), args["B"], args["H"], args["S"], args["D"], args["max_kv"],
                       args["block"], args["scale"], P(args["out"]),
                       P(args["lse"]) if args["lse"] else None,
                       P(args["ws"]) if args["ws"] else None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(D=64), binding.VSA_ERR_UNSUPPORTED),
    (dict(block=32), binding.VSA_ERR_UNSUPPORTED),
    (dict(S=100), binding.VSA_ERR_INVALID_ARG),           # not a multiple of the block
    (dict(S=64 * 4096), binding.VSA_ERR_UNSUPPORTED),     # more than VSA_MAX_BLOCKS blocks
    (dict(scale=0.0), binding.VSA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), binding.VSA_ERR_INVALID_ARG),
    (dict(B=-1), binding.VSA_ERR_INVALID_ARG),
])
def test_host_validation_without_gpu(lib, kw, code):
    assert _fwd(lib, **kw) == code


def test_empty_problem_is_a_no_op(lib):
    assert _fwd(lib, B=0) == binding.VSA_OK
    assert _fwd(lib, S=0) == binding.VSA_OK


def test_jenga_requires_square_blocks(lib):
    P = ctypes.c_void_p
    code = lib.jenga_fwd(P(1 << 20), P(2 << 20), P(3 << 20), P(4 << 20), 1, 1, 256, 128, 64, 128,
                         0.088, P(5 << 20), None, None, None)
    assert code == binding.VSA_ERR_UNSUPPORTED


def _gqa(lib, **kw):
    args = dict(B=1, Hq=4, Hkv=2, Sq=256, Sk=384, D=128, max_kv=4, block=64, vbs=6 << 20)
    args.update(kw)
    P = ctypes.c_void_p
    return lib.vsa_fwd_gqa(P(1 << 20), P(2 << 20), P(3 << 20), P(4 << 20), P(5 << 20),
                           P(args["vbs"]) if args["vbs"] else None, args["B"], args["Hq"],
                           args["Hkv"], args["Sq"], args["Sk"], args["D"], args["max_kv"],
                           args["block"], 0.088, P(7 << 20), None, None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(Hkv=3), binding.VSA_ERR_INVALID_ARG),           # Hq not a multiple of Hkv
    (dict(Hkv=0), binding.VSA_ERR_INVALID_ARG),
    (dict(Sk=100), binding.VSA_ERR_INVALID_ARG),          # Sk not a multiple of the block
    (dict(Sq=96), binding.VSA_ERR_INVALID_ARG),
    (dict(Sk=64 * 4096), binding.VSA_ERR_UNSUPPORTED),    # too many key blocks
    (dict(D=64), binding.VSA_ERR_UNSUPPORTED),
    (dict(max_kv=0), binding.VSA_ERR_CUDA),               # shape checks pass, then no device
])
def test_gqa_host_validation_without_gpu(lib, kw, code):
    got = _gqa(lib, **kw)
    if code == binding.VSA_ERR_CUDA:
        # without a GPU the device query fails first; with one, max_kv = 0 is rejected
        assert got in (binding.VSA_ERR_CUDA, binding.VSA_ERR_INVALID_ARG)
    else:
        assert got == code


def test_gqa_and_mask_empty_problems(lib):
    assert _gqa(lib, Sq=0) == binding.VSA_OK
    assert _gqa(lib, B=0) == binding.VSA_OK
    P = ctypes.c_void_p
    code = lib.vsa_fwd_from_mask(P(1 << 20), P(2 << 20), P(3 << 20), None, 0, None, 1, 2, 2, 0,
                                 256, 128, 64, 0.088, P(7 << 20), None, None, None)
    assert code == binding.VSA_OK
    code = lib.vsa_fwd_from_mask(P(1 << 20), P(2 << 20), P(3 << 20), P(4 << 20), 0, None, 1, 2,
                                 2, 256, 256, 128, 48, 0.088, P(7 << 20), None, None, None)
    assert code == binding.VSA_ERR_UNSUPPORTED


def _split(lib, splits=3, ws=8 << 20, ws_bytes=1 << 30, **kw):
    P = ctypes.c_void_p
    args = dict(B=1, Hq=2, Hkv=2, Sq=256, Sk=512, D=128, block=64)
    args.update(kw)
    return lib.vsa_fwd_split(P(1 << 20), P(2 << 20), P(3 << 20), P(4 << 20), P(5 << 20), None,
                             args["B"], args["Hq"], args["Hkv"], args["Sq"], args["Sk"],
                             args["D"], 4, args["block"], 0.088, splits, P(7 << 20), None,
                             P(ws) if ws else None, ws_bytes, None)


def test_split_validation(lib):
    assert _split(lib, splits=0) == binding.VSA_ERR_INVALID_ARG
    assert _split(lib, splits=binding.MAX_SPLITS + 1) == binding.VSA_ERR_INVALID_ARG
    assert _split(lib, D=64) == binding.VSA_ERR_UNSUPPORTED
    assert _split(lib, Sq=0) == binding.VSA_OK
    # 2 heads x 2 query blocks of 128 rows x 3 ranges, plus the scheduling counters
    n = lib.vsa_split_workspace_bytes(1, 2, 256, 64, 3)
    assert n == 256 + 2 * 2 * 3 * (128 * 128 + 3 * 128) * 4
    assert lib.vsa_split_workspace_bytes(1, 2, 100, 64, 3) == 0
    assert lib.vsa_split_workspace_bytes(1, 2, 256, 64, 0) == 0


def test_default_splits_fill_one_wave():
    """Split-KV ranges per item: the most that still give every (item, range) unit its own
    SM, 1 once the items fill the SMs, at most MAX_SPLITS."""
    # 24 heads of 128 query rows (one block-64 pair each) on 152 SMs: 6 ranges, 144 units
    assert binding.default_splits(1, 24, 128, 64, 152) == 6
    # block 128: one item per query block, 16 items
    assert binding.default_splits(2, 4, 256, 128, 152) == 9
    # the items already fill the SMs
    assert binding.default_splits(1, 152, 128, 64, 152) == 1
    assert binding.default_splits(1, 12, 16384, 64, 152) == 1
    # one item
    assert binding.default_splits(1, 1, 128, 64, 152) == binding.MAX_SPLITS
    assert binding.default_splits(1, 0, 128, 64, 152) == 1


def _bwd(lib, ws_bytes=1 << 30, **kw):
    P = ctypes.c_void_p
    args = dict(B=1, Hq=2, Hkv=1, Sq=256, Sk=512, D=128, block=64, max_kv=4)
    args.update(kw)
    return lib.vsa_bwd(P(1 << 20), P(2 << 20), P(3 << 20), P(4 << 20), P(5 << 20), P(6 << 20),
                       P(7 << 20), P(8 << 20), None, args["B"], args["Hq"], args["Hkv"],
                       args["Sq"], args["Sk"], args["D"], args["max_kv"], args["block"], 0.088,
                       P(9 << 20), P(10 << 20), P(11 << 20), P(12 << 20), ws_bytes, None)


def test_bwd_validation(lib):
    assert _bwd(lib, D=64) == binding.VSA_ERR_UNSUPPORTED
    assert _bwd(lib, block=32) == binding.VSA_ERR_UNSUPPORTED
    assert _bwd(lib, Hkv=3) == binding.VSA_ERR_INVALID_ARG
    assert _bwd(lib, Sk=100) == binding.VSA_ERR_INVALID_ARG
    assert _bwd(lib, B=0) == binding.VSA_OK
    # block map B*Hq*nbq*nbk bytes, -D and -lse per row, fp32 dq accumulator (each
    # 256-aligned)
    n = lib.vsa_bwd_workspace_bytes(1, 2, 256, 512, 64)
    assert n == 256 + 2 * 256 * 8 + 2 * 256 * 128 * 4
    assert lib.vsa_bwd_workspace_bytes(1, 2, 256, 500, 64) == 0
    # the step list holds a query block in 16 bits and a head of the group in 12
    assert _bwd(lib, Sq=64 * 65537, Hq=1) == binding.VSA_ERR_UNSUPPORTED
    assert _bwd(lib, Hq=4097, Hkv=1) == binding.VSA_ERR_UNSUPPORTED
    assert lib.vsa_bwd_workspace_bytes(1, 1, 64 * 65537, 512, 64) == 0


def test_metadata_validation(lib):
    P = ctypes.c_void_p
    assert lib.vsa_lut_to_bitmap(P(1 << 20), P(2 << 20), -1, 4, 8, P(3 << 20), None) == \
        binding.VSA_ERR_INVALID_ARG
    assert lib.vsa_lut_to_bitmap(P(1 << 20), P(2 << 20), 0, 4, 8, P(3 << 20), None) == binding.VSA_OK
    assert lib.vsa_bitmap_to_lut(P(1 << 20), 4, 8, 0, P(2 << 20), P(3 << 20), None) == \
        binding.VSA_ERR_INVALID_ARG
    assert lib.vsa_workspace_bytes() >= 8
