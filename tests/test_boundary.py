"""The C ABI boundary without a GPU: the library builds and loads, exports
every function include/aaren.h declares, and its host-only entry points
(sizes, strings, argument checks that fail before any CUDA call) behave."""
import ctypes
import os
import re

import pytest

from attention_prefix_scan_02_b300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "aaren.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(aaren_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def test_header_declares_the_abi():
    names = declared_functions()
    assert set(names) == set(binding.EXPORTS), names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(binding.LIB_PATH)
    for name in declared_functions():
        assert hasattr(raw, name), name


def test_status_strings(lib):
    for code in range(8):
        assert binding.status_string(code) and binding.status_string(code) != "unknown status"
    assert binding.status_string(99) == "unknown status"
    assert binding.aaren_abi_version() == 2


def test_binding_status_codes_match_the_header():
    text = open(HEADER).read()
    body = text[text.index("typedef enum {"):text.index("} aaren_status_t;")]
    codes = dict(re.findall(r"(AAREN_\w+)\s*=\s*(\d+)", body))
    assert codes, "no status codes found"
    for name, value in codes.items():
        assert getattr(binding, name) == int(value), name
    assert codes["AAREN_ERR_BOUNDS"] == "5"


def test_workspace_bytes(lib):
    assert binding.aaren_scan_workspace_bytes(1, 1, 0, 64) == 0
    assert binding.aaren_scan_workspace_bytes(0, 4, 100, 64) == 0
    assert binding.aaren_scan_workspace_bytes(1, 1, 10, 17) == 2 ** 64 - 1
    n1 = binding.aaren_scan_workspace_bytes(1, 16, 1 << 20, 128)
    C = min(binding.aaren_scan_chunk_tokens(128, binding.AAREN_F32),
            binding.aaren_scan_chunk_tokens(128, binding.AAREN_BF16))
    chunks = 16 * ((1 << 20) // C)
    assert n1 >= chunks * 2 * (128 + 4) * 4 + chunks * 4
    # grows with N
    assert binding.aaren_scan_workspace_bytes(1, 1, 1000, 64) < \
        binding.aaren_scan_workspace_bytes(1, 1, 100000, 64)


def test_chunk_tokens(lib):
    for d in (16, 32, 64, 128):
        for dt in (0, 1, 2):
            c = binding.aaren_scan_chunk_tokens(d, dt)
            assert c > 0 and c % 32 == 0
    assert binding.aaren_scan_chunk_tokens(48, 0) == 0
    assert binding.aaren_scan_chunk_tokens(64, 7) == 0


def test_argument_checks_before_any_cuda_call(lib):
    fake = ctypes.c_void_p(256)   # never dereferenced: each call fails its checks first
    # unsupported d and dtype
    assert lib.aaren_scan_forward(fake, fake, fake, fake, 1, 1, 8, 48, 0, None) == binding.AAREN_ERR_UNSUPPORTED
    assert lib.aaren_scan_forward(fake, fake, fake, fake, 1, 1, 8, 64, 9, None) == binding.AAREN_ERR_UNSUPPORTED
    # negative sizes, overflow
    assert lib.aaren_scan_forward(fake, fake, fake, fake, -1, 1, 8, 64, 0, None) == binding.AAREN_ERR_INVALID
    assert lib.aaren_scan_forward(fake, fake, fake, fake, 1 << 40, 1 << 20, 1 << 20, 64, 0,
                                  None) == binding.AAREN_ERR_INVALID
    # null pointers, misalignment, aliasing of O with K
    assert lib.aaren_scan_forward(None, fake, fake, fake, 1, 1, 8, 64, 0, None) == binding.AAREN_ERR_INVALID
    assert lib.aaren_scan_forward(fake, ctypes.c_void_p(260), fake, ctypes.c_void_p(1 << 20), 1, 1, 8, 64,
                                  0, None) == binding.AAREN_ERR_INVALID
    assert lib.aaren_scan_forward(fake, ctypes.c_void_p(4096), ctypes.c_void_p(1 << 20),
                                  ctypes.c_void_p(4096 + 256), 1, 1, 8, 64, 0, None) == binding.AAREN_ERR_INVALID
    # a partial state triple
    assert lib.aaren_scan_forward_ex(fake, fake, fake, fake, 1, 1, 8, 64, 0, fake, None, None,
                                     None, None, None, None, 0, None) == binding.AAREN_ERR_INVALID
    # step / init
    assert lib.aaren_step(fake, fake, fake, fake, fake, fake, fake, 4, 40, 0, None) == binding.AAREN_ERR_UNSUPPORTED
    assert lib.aaren_step(fake, fake, None, fake, fake, fake, fake, 4, 64, 0, None) == binding.AAREN_ERR_INVALID
    assert lib.aaren_state_init(fake, fake, fake, -3, 64, None) == binding.AAREN_ERR_INVALID
    # empty problems are no-ops that touch nothing
    assert lib.aaren_scan_forward(None, None, None, None, 0, 4, 8, 64, 0, None) == binding.AAREN_OK
    assert lib.aaren_step(None, None, None, None, None, None, None, 0, 64, 0, None) == binding.AAREN_OK
    assert lib.aaren_state_init(None, None, None, 0, 64, None) == binding.AAREN_OK


def test_debug_hook_is_host_state(lib):
    assert lib.aaren_debug_set_fault(5, 1000) == 0
    assert lib.aaren_debug_set_fault(-1, 0) == 0
    assert lib.aaren_debug_drop_arrival(3) == 0
    assert lib.aaren_debug_drop_arrival(-1) == 0


def test_no_cpu_fallback_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        binding.load(str(tmp_path / "missing.so"))


def test_product_code_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "attention_prefix_scan_02_b300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in text and "from oracle" not in text, fn
                assert "liboracle" not in text and "oracle.c" not in text, fn


def test_reduce_workspace_and_argument_checks(lib):
    # workspace: counters plus one state per part, parts bounded by the shape
    assert binding.aaren_reduce_workspace_bytes(0, 4, 100, 64) == 0
    assert binding.aaren_reduce_workspace_bytes(1, 1, 10, 17) == 2 ** 64 - 1
    one = binding.aaren_reduce_workspace_bytes(1, 1, 1, 64)
    assert one >= 256 + (64 + 4) * 4                       # N = 1: a single part
    big = binding.aaren_reduce_workspace_bytes(1, 16, 1 << 20, 128)
    assert (128 + 4) * 4 * 16 <= big <= 256 + 8192 * (128 + 4) * 4   # at most 8192 part states
    fake = ctypes.c_void_p(256)
    n = None
    # unsupported d / dtype; negative size; nothing requested; partial state
    assert lib.aaren_scan_reduce(fake, fake, fake, fake, 1, 1, 8, 48, 0, n, n, n, n, n, n, n, 0,
                                 n) == binding.AAREN_ERR_UNSUPPORTED
    assert lib.aaren_scan_reduce(fake, fake, fake, fake, 1, 1, 8, 64, 5, n, n, n, n, n, n, n, 0,
                                 n) == binding.AAREN_ERR_UNSUPPORTED
    assert lib.aaren_scan_reduce(fake, fake, fake, fake, 1, -1, 8, 64, 0, n, n, n, n, n, n, n, 0,
                                 n) == binding.AAREN_ERR_INVALID
    assert lib.aaren_scan_reduce(fake, fake, fake, n, 1, 1, 8, 64, 0, n, n, n, n, n, n, n, 0,
                                 n) == binding.AAREN_ERR_INVALID
    assert lib.aaren_scan_reduce(fake, fake, fake, fake, 1, 1, 8, 64, 0, n, n, n, fake, n, n, n, 0,
                                 n) == binding.AAREN_ERR_INVALID
    # the empty prefix has no output without a starting state
    assert lib.aaren_scan_reduce(fake, n, n, fake, 1, 1, 0, 64, 0, n, n, n, n, n, n, n, 0,
                                 n) == binding.AAREN_ERR_INVALID
    # misaligned K; o_last overlapping V
    assert lib.aaren_scan_reduce(fake, ctypes.c_void_p(260), fake, ctypes.c_void_p(1 << 20), 1, 1, 8,
                                 64, 0, n, n, n, n, n, n, n, 0, n) == binding.AAREN_ERR_INVALID
    assert lib.aaren_scan_reduce(fake, ctypes.c_void_p(1 << 20), ctypes.c_void_p(4096),
                                 ctypes.c_void_p(4096 + 256), 1, 1, 8, 64, 0, n, n, n, n, n, n, n,
                                 0, n) == binding.AAREN_ERR_INVALID
    # a workspace that is too small is refused before anything runs
    assert lib.aaren_scan_reduce(fake, fake, fake, ctypes.c_void_p(1 << 24), 1, 1, 8, 64, 0, n, n,
                                 n, n, n, n, ctypes.c_void_p(1 << 25), 16,
                                 n) == binding.AAREN_ERR_WORKSPACE
    # no heads: nothing to do
    assert lib.aaren_scan_reduce(n, n, n, fake, 0, 4, 8, 64, 0, n, n, n, n, n, n, n, 0,
                                 n) == binding.AAREN_OK


def test_linattn_argument_checks(lib):
    """aaren_linattn_forward rejects bad arguments before any CUDA call."""
    f = lib.aaren_linattn_forward
    ptr = 1 << 20   # never dereferenced: every case fails its checks first
    ok_args = dict(Q=ptr, K=ptr, V=ptr, O=ptr, B=1, H=1, N=8, d=64, M=8.0, pos0=0,
                   dtype=binding.AAREN_BF16, S_in=None, z_in=None, S_out=None, z_out=None)

    def call(**kw):
        a = dict(ok_args, **kw)
        return f(a["Q"], a["K"], a["V"], a["O"], a["B"], a["H"], a["N"], a["d"], a["M"],
                 a["pos0"], a["dtype"], a["S_in"], a["z_in"], a["S_out"], a["z_out"], None)

    assert call(d=32) == binding.AAREN_ERR_UNSUPPORTED
    assert call(d=128) == binding.AAREN_ERR_UNSUPPORTED
    assert call(dtype=binding.AAREN_F32) == binding.AAREN_ERR_UNSUPPORTED
    assert call(M=0.0) == binding.AAREN_ERR_INVALID
    assert call(M=-3.0) == binding.AAREN_ERR_INVALID
    assert call(M=float("inf")) == binding.AAREN_ERR_INVALID
    assert call(M=float("nan")) == binding.AAREN_ERR_INVALID
    assert call(pos0=-1) == binding.AAREN_ERR_INVALID
    assert call(N=-1) == binding.AAREN_ERR_INVALID
    assert call(S_in=ptr) == binding.AAREN_ERR_INVALID          # z_in missing
    assert call(S_out=ptr) == binding.AAREN_ERR_INVALID         # z_out missing
    assert call(S_in=ptr + 4, z_in=ptr) == binding.AAREN_ERR_INVALID   # misaligned state
    assert call(Q=None) == binding.AAREN_ERR_INVALID
    assert call(O=ptr + 8) == binding.AAREN_ERR_INVALID          # misaligned output
    assert call(B=0) == binding.AAREN_OK                         # nothing to do
    assert call(N=1 << 31) == binding.AAREN_ERR_INVALID          # beyond the 32-bit coordinates


def test_linattn_binding_rejects_host_tensors_and_bad_shapes():
    """The binding marshals only: it refuses host tensors (there is no CPU
    path) and mismatched shapes before calling the library."""
    import torch
    x = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        binding.aaren_linattn_forward(x, x, x, x.clone(), 8.0)
    with pytest.raises(ValueError, match="CUDA"):
        binding.linattn_forward(x, x, x)
