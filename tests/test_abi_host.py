"""Host-side tests of the C ABI that need no GPU: the library loads and exports every
declared entry point, and argument validation (sizes, alignment, the aliasing contract
of "feat(cuda): fuse activations and residual add into mmv f/q epilogues", What changed)
returns the documented status before anything is launched.  Pointers here are fake,
well-separated device addresses; no call below reaches a CUDA launch."""

import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "gemvfuse.h")
# fake, non-overlapping device addresses (validation never dereferences them)
W, X, A, D, S = (1 << 40), (2 << 40), (3 << 40), (4 << 40), (5 << 40)


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"GF_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_declares_the_abi():
    names = set(declared_functions())
    assert {"gemv_fused", "gemv_fused_ex", "gemv_glu", "fwht_signed", "gf_elementwise", "gf_dequantize",
            "gf_plan", "gf_plan_glu", "gf_device_status", "gf_status_string", "gf_last_cuda_error",
            "gf_version", "gf_prepare", "gf_prepare_glu", "gf_launch_prepared", "gf_free_prepared",
            "gf_graph_create", "gf_graph_launch", "gf_graph_free", "gemv_multi", "gf_prepare_multi",
            "gf_repair_count", "gf_copy", "gf_prepare_copy"} <= names


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    for name in declared_functions():
        assert hasattr(so, name), name


def test_library_hides_internal_symbols(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("nm not available")
    exported = {l.split()[-1] for l in out.stdout.splitlines() if " T " in l}
    assert set(declared_functions()) <= exported
    assert not any(n.startswith("_ZN2gf") for n in exported)


def test_status_strings(lib):
    assert lib.status_string(0) == "GF_OK"
    for s in (-1, -2, -3, -4, -5, -6):
        assert lib.status_string(s).startswith("GF_ERR_")
    assert lib.version() == 5


def g(lib, *a, **k):
    return lib.gemv_fused_ex(*a, check=False, stream=0, **k)


@pytest.mark.parametrize("args,kw,expect", [
    ((W, 7, X, 16, 32, 0, None, D), {}, -1),                    # bad weight type
    ((W, 0, X, 16, 32, 9, None, D), {}, -1),                    # bad epilogue
    ((W, 0, X, -1, 32, 0, None, D), {}, -1),                    # negative M
    ((W, 2, X, 16, 48, 0, None, D), {}, -3),                    # Q8_0 with K % 32 != 0
    ((W, 3, X, 16, 33, 0, None, D), {}, -3),                    # Q4_0 with K % 32 != 0
    ((W, 1, X, 16, 32, 0, None, D), {"ncols": 257}, -3),        # more than 256 columns
    ((W, 1, X, 16, 32, 0, None, D), {"ncols": -1}, -1),
    ((W, 1, X, 16, 32, 0, None, None), {}, -1),                 # null dst
    ((W, 1, X, 16, 32, 4, None, D), {}, -1),                    # ADD without operand
    ((W, 1, X, 16, 32, 3, None, D), {}, -1),                    # SILU_MUL without operand
    ((None, 1, X, 16, 32, 0, None, D), {}, -1),                 # null W
    ((W + 1, 1, X, 16, 32, 0, None, D), {}, -4),                # W not 2-byte aligned
    ((W + 2, 0, X, 16, 32, 0, None, D), {}, -4),                # F32 W not 4-byte aligned
    ((W, 1, X + 2, 16, 32, 0, None, D), {}, -4),                # x misaligned
    ((W, 1, X, 16, 32, 0, None, D + 1), {}, -4),                # dst misaligned
    ((W, 1, X, 16, 32, 0, None, W + 4), {}, -2),                # dst inside W
    ((W, 1, X, 16, 32, 0, None, X + 64), {}, -2),               # dst overlaps x
    ((W, 1, X, 16, 32, 4, A, A + 4), {}, -2),                   # dst partially overlaps aux
    ((W, 1, X, 16, 32, 3, A, A + 60), {}, -2),
    ((W, 1, X, 16, 32, 0, None, D), {"view": (4, 5)}, -1),      # view product != M
    ((W, 1, X, 16, 32, 0, None, D), {"view": (-4, 4)}, -1),
    ((W, 1, X, 16, 32, 0, None, D), {"fwht_signs": S, "fwht_block": 12, "nsigns": 12}, -1),
    ((W, 1, X, 16, 32, 0, None, D), {"fwht_signs": S, "fwht_block": 64, "nsigns": 64}, -1),   # K % B
    ((W, 1, X, 16, 16384, 0, None, D), {"fwht_signs": S, "fwht_block": 16384, "nsigns": 16384}, -3),
    ((W, 1, X, 16, 32, 0, None, D), {"fwht_signs": S, "fwht_block": 32, "nsigns": 0}, -1),
    ((W, 1, X, 16, 32, 0, None, D), {"fwht_signs": S, "fwht_block": 32, "nsigns": 5}, -1),
    ((W, 1, X, 16, 32, 0, None, S + 8), {"fwht_signs": S, "fwht_block": 32, "nsigns": 32}, -2),
    ((W, 1, X, 16, 32, 0, None, D), {"fwht_signs": S, "fwht_block": 32, "nsigns": 32,
                                     "fwht_workspace": (6 << 40) + 4}, -4),          # workspace misaligned
    ((W, 1, X, 16, 32, 0, None, D), {"fwht_signs": S, "fwht_block": 32, "nsigns": 32,
                                     "fwht_workspace": X + 64}, -2),                 # workspace over x
    ((W, 1, X, 16, 32, 0, None, D), {"fwht_signs": S, "fwht_block": 32, "nsigns": 32,
                                     "fwht_workspace": D}, -2),                      # workspace over dst
])
def test_gemv_validation(lib, args, kw, expect):
    assert g(lib, *args, **kw) == expect


def test_gemv_accepts_exact_in_place_and_empty(lib):
    # M == 0: nothing to launch, OK without touching the device
    assert g(lib, W, 1, X, 0, 32, 4, A, A) == 0
    assert g(lib, None, 1, None, 0, 0, 0, None, None) == 0
    # dst == aux exactly is allowed; plan says which kernel would run
    path, info = lib.plan(W, 1, X, 4096, 4096, 4, A, A, view=(32, 128))
    assert path == lib.PATH_STREAM and info["grid"] > 0
    # dst adjacent to (not overlapping) W is fine
    path, _ = lib.plan(W, 1, X, 16, 32, 0, None, W + 16 * 64)
    assert path in (lib.PATH_STREAM, lib.PATH_GENERIC)


@pytest.mark.parametrize("wt,K,w,expect_path", [
    (1, 4096, W, 1), (3, 4096, W, 1), (2, 4096, W, 1), (0, 512, W, 1),
    (1, 36, W, 2), (1, 4096, W + 2, 2), (3, 96, W, 2), (2, 224, W, 2), (0, 4, W, 2), (0, 8, W, 2),
    (0, 16, W, 1), (1, 24, W, 2),
])
def test_plan_path_selection(lib, wt, K, w, expect_path):
    path, info = lib.plan(w, wt, X, 1000, K, 0, None, D)
    assert path == expect_path
    if path == lib.PATH_STREAM:
        assert info["smem"] <= 232448 and 2 <= info["stages"] <= 8
        assert info["threads"] % 32 == 0 and info["threads"] <= 544


def test_plan_with_fwht_workspace_describes_the_plain_gemv(lib):
    path, info = lib.plan(W, 1, X, 5120, 5120, 4, A, A, ncols=8, fwht_signs=S, fwht_block=1024, nsigns=1024,
                          fwht_workspace=6 << 40)
    path2, info2 = lib.plan(W, 1, 6 << 40, 5120, 5120, 4, A, A, ncols=8)
    assert path == path2 == lib.PATH_TC and info == info2
    path, info = lib.plan(W, 1, X, 5120, 5120, 4, A, A, ncols=8, fwht_signs=S, fwht_block=1024, nsigns=1024,
                          fwht_workspace=6 << 40, tensor_cores=False)
    path2, info2 = lib.plan(W, 1, 6 << 40, 5120, 5120, 4, A, A, ncols=8, tensor_cores=False)
    assert path == path2 == lib.PATH_STREAM and info == info2


def test_plan_k_chunks_for_batches_and_long_rows(lib):
    _, info = lib.plan(W, 1, X, 5120, 5120, 4, A, A, ncols=8, fwht_signs=S, fwht_block=1024, nsigns=1024)
    assert info["k_chunk"] % 1024 == 0 and info["k_chunk"] < 5120
    _, info = lib.plan(W, 0, X, 4096, 14336, 0, None, D)
    assert info["k_chunk"] < 14336


@pytest.mark.parametrize("args,expect", [
    ((X, None, D, 100, 3), -1),        # block not a power of two
    ((X, None, D, 100, 64), -1),       # n % block
    ((X, None, D, 1 << 16, 32768), -3),
    ((X, S, D, 64, 32, 0), -1),        # nsigns 0
    ((X, S, D, 64, 32, 3), -1),        # n % nsigns
    ((X + 2, None, D, 64, 32), -4),
    ((X, None, X + 4, 64, 32), -2),    # partial overlap with x
    ((X, S, S, 64, 32, 32), -2),       # dst over the signs
    ((None, None, D, 64, 32), -1),
])
def test_fwht_validation(lib, args, expect):
    x, s, d, n, b = args[:5]
    ns = args[5] if len(args) > 5 else (32 if s else None)
    assert lib.fwht_signed(x, s, d, n, b, nsigns=ns, stream=0, check=False) == expect


def test_fwht_empty_is_ok(lib):
    assert lib.fwht_signed(None, None, None, 0, 1024, stream=0, check=False) == 0


@pytest.mark.parametrize("op,a,b,nb,d,n,expect", [
    (0, X, None, 1, D, 16, -1), (5, X, None, 1, D, 16, -1),
    (3, X, None, 16, D, 16, -1),            # MUL without b
    (4, X, A, 5, D, 16, -1),                # n % nb
    (1, X, None, 1, X + 4, 16, -2),         # partial overlap
    (4, X, A, 16, A + 8, 16, -2),
    (1, X + 1, None, 1, D, 16, -4),
])
def test_elementwise_validation(lib, op, a, b, nb, d, n, expect):
    assert lib.elementwise(op, a, b, d, n, nb=nb, stream=0, check=False) == expect


def test_dequantize_validation(lib):
    assert lib.dequantize(W, 9, 4, 32, D, stream=0, check=False) == -1
    assert lib.dequantize(W, 3, 4, 40, D, stream=0, check=False) == -3
    assert lib.dequantize(W, 3, 4, 32, W + 8, stream=0, check=False) == -2
    assert lib.dequantize(W + 1, 1, 4, 32, D, stream=0, check=False) == -4
    assert lib.dequantize(W, 1, 0, 32, D, stream=0, check=False) == 0


# ----------------------------------------------------------------------------- gated dual GEMV,
# RMS-normalisation prologue, split K
U2, GAM = (7 << 40), (8 << 40)


def glu(lib, *a, **k):
    return lib.gemv_glu(*a, check=False, stream=0, **k)


@pytest.mark.parametrize("args,kw,expect", [
    ((W, None, 1, X, 16, 32, D), {}, -1),                      # missing up matrix
    ((W, U2 + 1, 1, X, 16, 32, D), {}, -4),                    # up matrix misaligned
    ((W, U2, 1, X, 16, 32, U2 + 64), {}, -2),                  # dst inside the up matrix
    ((W, U2, 1, X, 16, 32, W + 64), {}, -2),                   # dst inside the gate matrix
    ((W, U2, 1, X, 16, 32, X), {}, -2),                        # dst over x
    ((W, U2, 7, X, 16, 32, D), {}, -1),                        # bad weight type
    ((W, U2, 1, X, 16, 32, D), {"ncols": 300}, -3),
    ((W, U2, 1, X, 16, 32, D), {"rms_norm_weight": GAM, "fwht_signs": S, "fwht_block": 32}, -3),
])
def test_glu_validation(lib, args, kw, expect):
    assert glu(lib, *args, **kw) == expect


def test_glu_empty_and_plan(lib):
    assert glu(lib, W, U2, 3, X, 0, 4096, D) == 0
    path, info = lib.plan_glu(W, U2, 3, X, 14336, 4096, D)
    assert path == lib.PATH_STREAM and info["split"] == 1
    assert info["stage_rows"] % 2 == 0  # every tile holds equal numbers of gate and up rows
    # unaligned up matrix (2-byte aligned f16) falls back to the generic kernel
    path, _ = lib.plan_glu(W, U2 + 2, 1, X, 64, 4096, D)
    assert path == lib.PATH_GENERIC


@pytest.mark.parametrize("kw,expect", [
    ({"rms_norm_weight": GAM + 2}, -4),                         # gamma misaligned
    ({"rms_norm_weight": GAM, "rms_norm_eps": -1.0}, -1),       # negative eps
    ({"rms_norm_weight": GAM, "rms_norm_eps": float("nan")}, -1),
    ({"rms_norm_weight": GAM, "rms_norm_eps": float("inf")}, -1),
    ({"rms_norm_weight": GAM, "fwht_signs": S, "fwht_block": 32, "nsigns": 32}, -3),  # two prologues
])
def test_rms_norm_validation(lib, kw, expect):
    assert g(lib, W, 1, X, 16, 32, 0, None, D, **kw) == expect


def test_rms_norm_dst_may_not_overlap_gamma(lib):
    assert g(lib, W, 1, X, 16, 32, 0, None, GAM + 4, rms_norm_weight=GAM) == -2


def test_rms_norm_plan(lib):
    path, _ = lib.plan(W, 1, X, 4096, 4096, 0, None, D, rms_norm_weight=GAM, rms_norm_eps=1e-6)
    assert path == lib.PATH_STREAM
    path, _ = lib.plan(W, 1, X, 4096, 4096, 0, None, D, rms_norm_weight=GAM + 4, rms_norm_eps=1e-6)
    assert path == lib.PATH_GENERIC  # gamma not 16-byte aligned


@pytest.mark.parametrize("M,K,wt,expect_split", [
    (32, 4096, 3, 1),      # the 32-row sigmoid projection: 18 KB per CTA, not worth a cluster
    (32, 32768, 3, 4),     # 128 KB of x + 18 KB of weights per CTA: 4 CTAs per row range
    (16, 65536, 1, 8),
    (8, 131072, 1, 8),
    (76, 32768, 1, 2),
    (77, 32768, 1, 1),     # more than half the SMs' worth of rows: no split
    (32, 16384, 1, 1),     # 96 KB per CTA
    (4096, 4096, 1, 1),
])
def test_split_k_selection(lib, M, K, wt, expect_split):
    path, info = lib.plan(W, wt, X, M, K, 0, None, D)
    assert path == lib.PATH_STREAM and info["split"] == expect_split
    assert info["grid"] % expect_split == 0 and info["grid"] <= 152
    if expect_split > 1:
        assert info["k_chunk"] * (expect_split - 1) < K
    _, off = lib.plan(W, wt, X, M, K, 0, None, D, split_k=False)
    assert off["split"] == 1


def test_split_k_with_glu_and_prologues(lib):
    _, info = lib.plan_glu(W, U2, 3, X, 32, 32768, D)
    assert info["split"] == 4
    _, info = lib.plan(W, 1, X, 32, 40960, 0, None, D, fwht_signs=S, fwht_block=1024, nsigns=1024)
    assert info["split"] == 4 and info["k_chunk"] % 1024 == 0
    _, info = lib.plan(W, 1, X, 32, 32768, 0, None, D, rms_norm_weight=GAM)
    assert info["split"] == 4
    # a batch multiplies the x bytes each CTA streams
    _, info = lib.plan(W, 3, X, 32, 8192, 0, None, D, ncols=4)
    assert info["split"] == 4


# ----------------------------------------------------------------------------- Q4_K

def test_q4_k_validation_and_plan(lib):
    assert lib.Q4_K == 4
    assert g(lib, W, lib.Q4_K, X, 16, 4096 + 32, 0, None, D) == -3     # K % 256
    assert g(lib, W, 5, X, 16, 4096, 0, None, D) == -1                  # past the last format
    path, info = lib.plan(W, lib.Q4_K, X, 4096, 4096, 0, None, D)
    assert path == lib.PATH_STREAM and info["k_chunk"] == 4096
    path, _ = lib.plan(W + 2, lib.Q4_K, X, 4096, 4096, 0, None, D)
    assert path == lib.PATH_GENERIC                                     # rows not 16-byte aligned
    path, info = lib.plan(W, lib.Q4_K, X, 4096, 14336, 4, A, A, ncols=8)
    assert path == lib.PATH_STREAM and info["k_chunk"] % 256 == 0
    assert lib.dequantize(W, lib.Q4_K, 4, 300, D, stream=0, check=False) == -3
    assert lib.dequantize(W, 6, 4, 256, D, stream=0, check=False) == -1


def test_wide_batch_validation_covers_every_column(lib):
    # 20 columns: dst overlapping x anywhere in the whole batch is refused
    assert g(lib, W, 1, X, 16, 32, 0, None, X + 19 * 32 * 4, ncols=20) == -2
    path, info = lib.plan(W, 3, X, 4096, 4096, 4, A, A, ncols=20)
    path8, info8 = lib.plan(W, 3, X, 4096, 4096, 4, A, A, ncols=8)
    assert path == path8 == lib.PATH_STREAM and info == info8  # each block's launch
    # tensor cores: blocks of 16 columns
    _, i100 = lib.plan(W, 1, X, 4096, 4096, 4, A, A, ncols=100)   # 6 blocks of 16, then 4
    _, i16 = lib.plan(W, 1, X, 4096, 4096, 4, A, A, ncols=16)
    assert i100 == i16


# ----------------------------------------------------------------------------- tensor-core path

@pytest.mark.parametrize("M,K,ncols,expect_split", [
    (5120, 5120, 8, 3),     # 40 row tiles: 3 CTAs per tile
    (4096, 4096, 8, 4),     # 32 tiles
    (14336, 4096, 16, 1),   # 112 tiles
    (100, 4096, 4, 8),      # one ragged tile
    (4096, 64, 8, 1),       # one K stage
])
def test_tc_plan(lib, M, K, ncols, expect_split):
    path, info = lib.plan(W, 1, X, M, K, 0, None, D, ncols=ncols)
    assert path == lib.PATH_TC and info["split"] == expect_split
    assert info["grid"] == -(-M // 128) * expect_split and info["grid"] <= 152
    assert info["smem"] <= 232448 and 2 <= info["stages"] <= 12 and info["threads"] == 192


@pytest.mark.parametrize("kw,args", [
    ({"ncols": 1}, (W, 1, X, 4096, 4096)),                  # one column: CUDA cores
    ({"ncols": 2}, (W, 1, X, 4096, 4096)),                  # below the tensor-core batch
    ({"ncols": 8}, (W, 3, X, 4096, 4096)),                  # block formats: CUDA cores
    ({"ncols": 8}, (W, 1, X, 4096, 4096 + 32)),             # K % 64
    ({"ncols": 8}, (W + 2, 1, X, 4096, 4096)),              # W not 16-byte aligned
    ({"ncols": 8, "tensor_cores": False}, (W, 1, X, 4096, 4096)),
    ({"ncols": 8, "fwht_signs": S, "fwht_block": 1024, "nsigns": 1024}, (W, 1, X, 4096, 4096)),  # on-chip prologue
    ({"ncols": 8, "rms_norm_weight": 8 << 40}, (W, 1, X, 4096, 4096)),
])
def test_tc_not_chosen(lib, kw, args):
    path, _ = lib.plan(*args, 0, None, D, **kw)
    assert path in (lib.PATH_STREAM, lib.PATH_GENERIC)


@pytest.mark.parametrize("M,split", [(10240, 1), (8192, 2), (5184, 3), (4196, 4), (3800, 5), (3100, 6),
                                     (2600, 7), (1000, 8)])
@pytest.mark.parametrize("ncols", [3, 8, 13, 16])
def test_tc_plan_split_sizes(lib, M, split, ncols):
    """F16 batches of 3..16 columns plan onto the tensor cores; K is split over a cluster
    of SMs // tiles CTAs (at most 8; without a device no residency limit lowers it), the
    grid fits the 152 SMs at once, and the shared memory fits a CTA."""
    path, info = lib.plan(W, 1, X, M, 1024, 4, A, A, ncols=ncols)
    tiles = -(-M // 128)
    assert path == lib.PATH_TC
    assert info["split"] == split == min(8, 152 // tiles)
    assert info["grid"] == tiles * split <= 152
    assert info["threads"] == 192 and 3 <= info["stages"] <= 12 and info["smem"] <= 232448


@pytest.mark.parametrize("dst,src,nbytes,expect", [
    (D, X, -16, -1),            # negative size
    (D, X, 40, -1),             # not a multiple of 16
    (None, X, 64, -1),          # null destination
    (D, None, 64, -1),          # null source
    (D + 8, X, 64, -4),         # destination not 16-byte aligned
    (D, X + 4, 64, -4),         # source not 16-byte aligned
    (X + 32, X, 64, -2),        # overlapping ranges
    (D, X, 0, 0),               # nothing to copy: OK, nothing launched
    (None, None, 0, 0),
])
def test_copy_validation(lib, dst, src, nbytes, expect):
    assert lib.copy(dst, src, nbytes, stream=0, check=False) == expect
    if expect != 0:  # (a valid handle needs a current device)
        assert lib.prepare_copy(dst, src, nbytes, check=False) == expect


def test_selftest_wait_validation(lib):
    assert lib.selftest_wait_timeout(0, D, stream=0, check=False) == -1
    assert lib.selftest_wait_timeout(2000000, D, stream=0, check=False) == -1
    assert lib.selftest_wait_timeout(1000, None, stream=0, check=False) == -1
    assert lib.selftest_wait_timeout(1000, D + 2, stream=0, check=False) == -4


# ----------------------------------------------------------------------------- prepared calls

def test_prepare_validates_like_the_direct_call(lib):
    # the same status as gemv_fused_ex, before anything is planned; no handle is returned
    h = ctypes.c_void_p(123)
    st = lib.raw.gf_prepare(ctypes.c_void_p(W), 9, ctypes.c_void_p(X), 64, 256, 0, None, ctypes.c_void_p(D),
                            None, ctypes.byref(h))
    assert st == lib.ERR_INVALID and not h.value
    st = lib.raw.gf_prepare(ctypes.c_void_p(W), 1, ctypes.c_void_p(X), 64, 256, 0, None, ctypes.c_void_p(W + 64),
                            None, ctypes.byref(h))  # dst inside W
    assert st == lib.ERR_ALIAS and not h.value
    st = lib.raw.gf_prepare(ctypes.c_void_p(W), 1, ctypes.c_void_p(X), 64, 256, 4, None, ctypes.c_void_p(D),
                            None, ctypes.byref(h))  # ADD without its operand
    assert st == lib.ERR_INVALID and not h.value
    st = lib.raw.gf_prepare_glu(ctypes.c_void_p(W), ctypes.c_void_p(A), 1, ctypes.c_void_p(X), 64, 256,
                                ctypes.c_void_p(W + 64), None, ctypes.byref(h))
    assert st == lib.ERR_ALIAS and not h.value
    # no place for the handle
    assert lib.raw.gf_prepare(ctypes.c_void_p(W), 1, ctypes.c_void_p(X), 64, 256, 0, None, ctypes.c_void_p(D),
                              None, None) == lib.ERR_INVALID


def test_launch_prepared_arguments(lib):
    arr = (ctypes.c_void_p * 2)(None, None)
    assert lib.raw.gf_launch_prepared(arr, 0, None) == lib.OK  # nothing to launch
    assert lib.raw.gf_launch_prepared(None, 1, None) == lib.ERR_INVALID
    assert lib.raw.gf_launch_prepared(arr, -1, None) == lib.ERR_INVALID
    lib.raw.gf_free_prepared(None)  # ignored


def test_graph_arguments(lib):
    h = ctypes.c_void_p(7)
    arr = (ctypes.c_void_p * 1)(None)
    assert lib.raw.gf_graph_create(arr, 0, ctypes.byref(h)) == lib.ERR_INVALID and not h.value
    assert lib.raw.gf_graph_create(arr, 1, ctypes.byref(h)) == lib.ERR_INVALID and not h.value  # NULL handle
    assert lib.raw.gf_graph_create(arr, 1, None) == lib.ERR_INVALID
    assert lib.raw.gf_graph_launch(None, None) == lib.ERR_INVALID
    lib.raw.gf_graph_free(None)  # ignored


# ----------------------------------------------------------------------------- several matrices, one x

def _items(lib, *specs):
    arr = (lib.MultiItem * len(specs))()
    for i, (w, m, e, a, d) in enumerate(specs):
        arr[i].W, arr[i].M, arr[i].epilogue, arr[i].aux, arr[i].dst = w, m, e, a, d
    return arr


def test_gemv_multi_validation(lib):
    f = lib.raw.gemv_multi
    K, M = 256, 64
    ok_items = _items(lib, (W, M, 0, None, D), (W + (1 << 30), M, 1, None, D + (1 << 30)))
    assert f(None, 1, 1, ctypes.c_void_p(X), K, None, None) == lib.ERR_INVALID
    assert f(ok_items, 0, 1, ctypes.c_void_p(X), K, None, None) == lib.ERR_INVALID
    five = _items(lib, *[(W + (i << 30), M, 0, None, D + (i << 30)) for i in range(5)])
    assert f(five, 5, 1, ctypes.c_void_p(X), K, None, None) == lib.ERR_UNSUPPORTED
    # a matrix that is invalid alone (ADD without its operand)
    bad = _items(lib, (W, M, 0, None, D), (W + (1 << 30), M, 4, None, D + (1 << 30)))
    assert f(bad, 2, 1, ctypes.c_void_p(X), K, None, None) == lib.ERR_INVALID
    # one item's dst over another item's W, or over another item's dst
    cross = _items(lib, (W, M, 0, None, D), (W + (1 << 30), M, 0, None, W + 64))
    assert f(cross, 2, 1, ctypes.c_void_p(X), K, None, None) == lib.ERR_ALIAS
    same = _items(lib, (W, M, 0, None, D), (W + (1 << 30), M, 0, None, D + 4 * (M // 2)))
    assert f(same, 2, 1, ctypes.c_void_p(X), K, None, None) == lib.ERR_ALIAS
    # a dst view has no meaning for several outputs
    o = lib.make_opts(view=(8, 8))
    assert f(ok_items, 2, 1, ctypes.c_void_p(X), K, ctypes.byref(o), None) == lib.ERR_INVALID
    h = ctypes.c_void_p(5)
    assert lib.raw.gf_prepare_multi(cross, 2, 1, ctypes.c_void_p(X), K, None, ctypes.byref(h)) == lib.ERR_ALIAS
    assert not h.value
