"""Host-side checks of the C ABI (no GPU needed): the library builds, loads,
exports every entry point declared in include/nvfp4moe.h, and its pure host
functions (sizes, status strings, argument validation) behave as declared."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4moe.h")


@pytest.fixture(scope="session")
def lib():
    from nvfp4_block_scaled_07_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?((?:moe|nvfp4moe)_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_layer_calls():
    names = declared_functions()
    for n in ["moe_route_topk", "moe_quantize_nvfp4", "moe_permute", "moe_grouped_gemm_nvfp4", "moe_finalize"]:
        assert n in names
    assert len(names) >= 16


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version(lib):
    lib.nvfp4moe_status_string.restype = ctypes.c_char_p
    for s in range(8):
        assert lib.nvfp4moe_status_string(s).decode()
    assert lib.nvfp4moe_status_string(99).decode() == "unknown status"
    assert lib.nvfp4moe_version() >= 10000


def test_size_queries(lib):
    lib.nvfp4moe_blocked_scales_bytes.restype = ctypes.c_size_t
    lib.nvfp4moe_blocked_scales_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
    assert lib.nvfp4moe_blocked_scales_bytes(1, 64) == 128 * 4
    assert lib.nvfp4moe_blocked_scales_bytes(129, 6144) == 256 * 384
    assert lib.nvfp4moe_blocked_scales_bytes(10, 100) == 0
    lib.moe_permute_rows_capacity.restype = ctypes.c_int64
    # each expert may add up to 127 padding rows; capacity is a multiple of 128
    assert lib.moe_permute_rows_capacity(128, 256, 8) == ((1024 + 256 * 127 + 127) // 128) * 128
    assert lib.moe_permute_rows_capacity(16, 8, 2) % 128 == 0
    lib.moe_permute_workspace_size.restype = ctypes.c_size_t
    assert lib.moe_permute_workspace_size(16384, 64, 8) >= 16384 * 8 * 4
    # tiled weights: (rows / 128) * ceil(K / 256) boxes of 128 x 128 bytes
    lib.nvfp4moe_tiled_weights_bytes.restype = ctypes.c_size_t
    lib.nvfp4moe_tiled_weights_bytes.argtypes = [ctypes.c_int64, ctypes.c_int]
    assert lib.nvfp4moe_tiled_weights_bytes(256 * 4096, 6144) == (256 * 4096 // 128) * 24 * 16384
    assert lib.nvfp4moe_tiled_weights_bytes(128, 320) == 2 * 16384        # a partial last K chunk is padded
    assert lib.nvfp4moe_tiled_weights_bytes(128, 6144) == 128 * 6144 // 2  # no padding when K % 256 == 0
    assert lib.nvfp4moe_tiled_weights_bytes(100, 256) == 0
    assert lib.nvfp4moe_tiled_weights_bytes(128, 96) == 0
    lib.moe_quantize_nvfp4_workspace_size.restype = ctypes.c_size_t
    lib.moe_quantize_nvfp4_workspace_size.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int]
    assert lib.moe_quantize_nvfp4_workspace_size(4, 64, 0) == 0
    assert lib.moe_quantize_nvfp4_workspace_size(4, 64, 1) >= 4


def test_argument_validation_before_any_device_work(lib):
    _no_device()
    p = ctypes.c_void_p
    lib.moe_route_topk.argtypes = [p, p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, p, p, p]
    assert lib.moe_route_topk(None, None, 4, 2048, 2, 1, 1, None, None, None) == 2    # E > 1024
    assert lib.moe_route_topk(None, None, 4, 8, 9, 1, 1, None, None, None) == 2       # k > E
    assert lib.moe_route_topk(None, None, 4, 8, 2, 7, 1, None, None, None) == 1       # bad score_fn
    assert lib.moe_route_topk(None, None, 0, 8, 2, 1, 1, None, None, None) == 0       # T = 0 is a no-op
    g = lib.moe_grouped_gemm_nvfp4
    g.argtypes = [p, p, p, p, p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, p, p, p, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, p, p, p, ctypes.c_int, ctypes.c_int, p, ctypes.c_size_t, p]
    dummy = p(256)
    assert g(dummy, dummy, dummy, dummy, dummy, 8, 1024, 32, dummy, dummy, dummy, 256, 100, 0, None, dummy, None, 0,
             0, None, 0, None) == 2      # K % 64 != 0
    assert g(dummy, dummy, dummy, dummy, dummy, 8, 1024, 32, dummy, dummy, dummy, 384, 256, 1, dummy, dummy, dummy, 0,
             0, None, 0, None) == 2      # SwiGLU N % 256 != 0
    assert g(dummy, dummy, dummy, dummy, dummy, 8, 1000, 32, dummy, dummy, dummy, 256, 256, 0, None, dummy, None, 0,
             0, None, 0, None) == 1      # rows_capacity % 128 != 0
    assert g(dummy, dummy, dummy, dummy, dummy, 8, 1024, 32, dummy, dummy, dummy, 256, 256, 7, None, dummy, None, 0,
             0, None, 0, None) == 1      # bad epilogue
    assert g(dummy, dummy, dummy, dummy, dummy, 8, 1024, 32, dummy, dummy, dummy, 256, 256, 1, None, dummy, None, 0,
             0, None, 0, None) == 1      # SWIGLU_NVFP4 without its scale pointers
    assert g(dummy, dummy, dummy, dummy, dummy, 8, 1024, 32, dummy, dummy, dummy, 256, 256, 0, None, dummy, None, 0,
             5, None, 0, None) == 1      # unknown weight layout
    assert g(dummy, dummy, dummy, dummy, dummy, 8, 1024, 32, dummy, dummy, dummy, 384, 256, 0, None, dummy, None, -1,
             0, None, 0, None) == 2      # token-major tiles need N % 256 == 0
    t = lib.nvfp4moe_tile_weights
    t.argtypes = [p, ctypes.c_int64, ctypes.c_int, p, p]
    assert t(dummy, 100, 256, dummy, None) == 2     # rows % 128
    assert t(dummy, 128, 96, dummy, None) == 2      # K % 64
    assert t(p(8), 128, 256, dummy, None) == 1      # misaligned
    q = lib.moe_quantize_nvfp4
    q.argtypes = [p, ctypes.c_int64, ctypes.c_int64, p, ctypes.c_int, p, p, p, ctypes.c_size_t, p]
    assert q(dummy, 4, 40, dummy, 0, dummy, dummy, None, 0, None) == 2     # cols % 16
    assert q(dummy, 4, 96, dummy, 2, dummy, dummy, None, 0, None) == 2     # blocked needs cols % 64
    assert q(dummy, 4, 64, dummy, 1, dummy, dummy, None, 0, None) == 4     # global amax needs workspace
    assert q(p(8), 4, 64, dummy, 0, dummy, dummy, None, 0, None) == 1      # misaligned x


def test_binding_imports_and_names_match_header():
    from nvfp4_block_scaled_07_gb300 import binding
    for n in ["moe_route_topk", "moe_quantize_nvfp4", "moe_permute", "moe_grouped_gemm_nvfp4", "moe_finalize",
              "moe_scales_to_blocked"]:
        assert callable(getattr(binding, n))


def test_untile_weights_inverts_the_documented_tiling():
    """The test utility that reads tiled weights back (used against the
    oracle's codes on the GPU) inverts the layout the header defines, checked
    against a direct box-by-box construction."""
    import numpy as np
    from tests import nvfp4_testutil as U
    rng = np.random.default_rng(3)
    for E, N, K in [(2, 128, 320), (3, 256, 512), (1, 128, 64), (2, 384, 768)]:
        w = rng.integers(0, 256, size=(E, N, K // 2), dtype=np.uint8)
        kc = (K + 255) // 256
        tiled = np.zeros(E * N // 128 * kc * 16384, np.uint8)
        rows = w.reshape(E * N, K // 2)
        for rb in range(E * N // 128):
            for c in range(kc):
                base = (rb * kc + c) * 16384
                for r in range(128):
                    seg = rows[rb * 128 + r, c * 128:c * 128 + 128]
                    tiled[base + r * 128:base + r * 128 + len(seg)] = seg
        np.testing.assert_array_equal(U.untile_weights(tiled, E, N, K), w)


def test_binding_fails_loudly_without_the_library(tmp_path):
    """A copy of the package without libnvfp4moe.so does not import: there is
    no fallback implementation to run instead."""
    import shutil
    import subprocess
    import sys
    src = os.path.join(ROOT, "nvfp4_block_scaled_07_gb300")
    dst = tmp_path / "nvfp4_block_scaled_07_gb300"
    dst.mkdir()
    for name in ("__init__.py", "binding.py", "workloads.py"):
        shutil.copy(os.path.join(src, name), dst / name)
    r = subprocess.run([sys.executable, "-c", "import nvfp4_block_scaled_07_gb300.binding"], cwd=tmp_path,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode != 0
    assert "ImportError" in r.stderr and "no fallback" in r.stderr


def test_binding_rejects_host_tensors():
    """Host (CPU) tensors are refused before any call into the library, so a
    caller cannot end up with a host computation."""
    import torch
    from nvfp4_block_scaled_07_gb300 import binding as B
    with pytest.raises(ValueError, match="CUDA tensor"):
        B.moe_route_topk(torch.zeros(4, 8), 2)
    with pytest.raises(ValueError, match="CUDA tensor"):
        B.moe_quantize_nvfp4(torch.zeros(4, 64, dtype=torch.bfloat16))
    with pytest.raises(TypeError):
        B.moe_quantize_nvfp4(torch.zeros(4, 64, dtype=torch.float64))


def test_grouped_gemm_binding_requires_the_routed_row_count():
    """The padded capacity would always pick token-major tiles, so the binding
    asks for the routed rows instead of guessing them."""
    import torch
    from nvfp4_block_scaled_07_gb300 import binding as B
    with pytest.raises(ValueError, match="m_total"):
        B.moe_grouped_gemm_nvfp4(*([torch.zeros(1)] * 8))
    with pytest.raises(ValueError, match="m_total"):
        B.moe_grouped_gemm_mxfp4(*([torch.zeros(1)] * 6))


@pytest.mark.parametrize("rows,cols,block", [(1, 64, 16), (130, 320, 16), (256, 1024, 16), (5, 128, 32),
                                             (300, 640, 32)])
def test_blocked_layout_helper_follows_the_header(lib, rows, cols, block):
    """The test utility that reads the library's blocked scales, against the
    layout as the header states it, written out loop by loop: 128-row x
    (4 * block)-element groups of 512 bytes at (rb * groups_per_row + kb) *
    512, row r of a group at (r % 32) * 16 + (r / 32) * 4, then the scale's
    index within its group of four.  Every byte of the buffer is addressed
    exactly once, and the buffer size is the library's."""
    import numpy as np
    from tests import nvfp4_testutil as U
    rp = -(-rows // 128) * 128
    per_row = cols // block
    groups = cols // (4 * block)
    idx = U.blocked_index(rp, cols, block)
    for r in range(rp):
        for j in range(per_row):
            rb, kb, rr = r // 128, j // 4, r % 128
            assert idx[r, j] == (rb * groups + kb) * 512 + (rr % 32) * 16 + (rr // 32) * 4 + j % 4
    assert sorted(idx.ravel().tolist()) == list(range(rp * per_row))
    q = lib.nvfp4moe_blocked_scales_bytes if block == 16 else lib.nvfp4moe_mxfp4_blocked_scales_bytes
    q.restype = ctypes.c_size_t
    q.argtypes = [ctypes.c_int64, ctypes.c_int64]
    assert q(rows, cols) == rp * per_row


def _header_signatures():
    """{name: (return kind, [argument kinds])} from the header's declarations;
    kinds: p (pointer), i (int), u32 (uint32_t), i64 (int64_t), sz (size_t), cstr (const char*)."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    text = re.sub(r"^\s*#.*$", "", text, flags=re.M)

    def kind(decl):
        decl = decl.strip()
        if decl in ("", "void"):
            return None
        if "*" in decl or decl.startswith("cudaStream_t"):
            return "cstr" if decl.replace(" ", "").startswith("constchar*") and "(" not in decl else "p"
        t = decl.split()[0] if not decl.startswith("const ") else decl.split()[1]
        return {"int": "i", "int32_t": "i", "uint32_t": "u32", "int64_t": "i64", "size_t": "sz"}[t]

    sigs = {}
    for m in re.finditer(r"([\w\s\*]+?)\b((?:moe|nvfp4moe)_\w+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
        ret = m.group(1).split("\n")[-1].strip()
        args = [kind(a) for a in m.group(3).split(",")]
        sigs[m.group(2)] = (kind(ret + " x") if "*" not in ret else "cstr", [a for a in args if a])
    return sigs


def test_binding_signatures_match_the_header():
    """Every ctypes signature in the binding has the header's argument count
    and kinds (a pointer, an int, an int64_t or a size_t in each place), so a
    call can never shift its arguments."""
    from nvfp4_block_scaled_07_gb300 import binding as B
    kinds = {ctypes.c_void_p: "p", ctypes.c_int: "i", ctypes.c_uint32: "u32", ctypes.c_int64: "i64",
             ctypes.c_size_t: "sz", ctypes.c_char_p: "cstr"}
    hdr = _header_signatures()
    assert set(B._SIGS) == set(hdr), set(B._SIGS) ^ set(hdr)
    for name, (res, args) in B._SIGS.items():
        h_res, h_args = hdr[name]
        assert [kinds[a] for a in args] == h_args, name
        assert kinds[res] == h_res, name


def _no_device():
    """These cases pass dummy pointers: each must be refused (or be a no-op)
    before any device work, so they run only where no GPU could be touched."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("host-validation cases with dummy pointers run only without a GPU")


def test_validation_of_the_other_calls(lib):
    _no_device()
    p = ctypes.c_void_p
    dummy = p(256)
    r = lib.moe_route_topk
    r.argtypes = [p, p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, p, p, p]
    assert r(dummy, None, 4, 8, 9, 1, 1, dummy, dummy, None) == 2        # k > E
    assert r(dummy, None, 4, 2048, 8, 1, 1, dummy, dummy, None) == 2     # E > 1024
    assert r(dummy, None, 4, 64, 33, 1, 1, dummy, dummy, None) == 2      # k > 32
    assert r(dummy, None, 4, 8, 2, 7, 1, dummy, dummy, None) == 1        # unknown score function
    assert r(dummy, None, -1, 8, 2, 1, 1, dummy, dummy, None) == 1       # T < 0
    assert r(None, None, 4, 8, 2, 1, 1, dummy, dummy, None) == 1         # null logits
    q = lib.moe_quantize_nvfp4
    q.argtypes = [p, ctypes.c_int64, ctypes.c_int64, p, ctypes.c_int, p, p, p, ctypes.c_size_t, p]
    assert q(dummy, 4, 40, dummy, 0, dummy, dummy, None, 0, None) == 2   # cols % 16
    assert q(dummy, 4, 48, dummy, 2, dummy, dummy, None, 0, None) == 2   # blocked scales need cols % 64
    assert q(dummy, 4, 64, dummy, 8, dummy, dummy, None, 0, None) == 1   # unknown flag
    assert q(p(258), 4, 64, dummy, 0, dummy, dummy, None, 0, None) == 1  # misaligned x
    assert q(dummy, 4, 64, dummy, 1, dummy, dummy, None, 0, None) == 4   # global scale needs its workspace
    f = lib.moe_finalize
    f.argtypes = [p, p, p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, p, p]
    assert f(dummy, dummy, dummy, 4, 2, 12, 1024, dummy, None) == 2      # H % 8
    assert f(dummy, dummy, dummy, 4, 0, 16, 1024, dummy, None) == 1      # k < 1
    assert f(p(264), dummy, dummy, 4, 2, 16, 1024, dummy, None) == 1     # misaligned y
    pr = lib.moe_permute
    pr.argtypes = [p, ctypes.c_int, ctypes.c_int, ctypes.c_int, p, p, ctypes.c_int] + [p] * 7 + [p, ctypes.c_size_t, p]
    args = [dummy] * 7
    assert pr(dummy, 4, 8, 2, dummy, dummy, 100, *args, dummy, 1 << 20, None) == 2    # H % 64
    assert pr(dummy, 4, 8, 9, dummy, dummy, 128, *args, dummy, 1 << 20, None) == 2    # k > E
    assert pr(dummy, 4, 8, 2, dummy, dummy, 128, *args, dummy, 4, None) == 4          # workspace too small
    # empty batches are no-ops that touch nothing, also with null buffers
    assert r(None, None, 0, 8, 2, 1, 1, None, None, None) == 0
    assert q(None, 0, 64, None, 1, None, None, None, 0, None) == 0
    assert f(None, None, None, 0, 2, 16, 0, None, None) == 0


def test_gemm_tile_choice_follows_rows_per_expert(lib):
    """The automatic tile orientation (host logic, no device): weight rows as
    M below 64 routed rows per expert on average, token-major from 64,
    token-major on CTA pairs from 512; an explicit tile_n or an N that is not
    a multiple of 256 is kept."""
    f = lib.nvfp4moe_gemm_tile_choice
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int]
    assert f(256, 4096, 1024, 0) == 0            # decode_t128: 4 rows per expert
    assert f(256, 4096, 16383, 0) == 0
    assert f(256, 4096, 16384, 0) == -1          # skewed_t2048: 64 rows per expert on average
    assert f(64, 8192, 32767, 0) == -1
    assert f(64, 8192, 32768, 0) == -2           # 512 rows per expert
    assert f(64, 8192, 131072, 0) == -2          # prefill_t16384
    assert f(64, 8192, 131072, 128) == 128       # explicit choice kept
    assert f(64, 8192, 131072, -1) == -1
    assert f(64, 384, 131072, 0) == 0            # N % 256 != 0: no token-major tiles
