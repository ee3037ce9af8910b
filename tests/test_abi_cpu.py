"""CPU-only checks of the C ABI: the library builds, loads and exports every
function the header declares; host-side validation rejects bad arguments
before any CUDA call (so these run without a GPU)."""
import ctypes
import glob
import os
import re

import pytest

from gathered_rank_gemm_gb300 import binding
from gathered_rank_gemm_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return binding.load()


def declared_functions():
    text = "".join(open(h).read() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lora_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("lora_prepare_metadata", "lora_shrink", "lora_expand", "lora_workspace_size",
              "lora_read_status", "lora_error_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported"
    assert set(binding.EXPORTED) <= set(declared_functions())


def test_only_the_abi_is_exported():
    out = os.popen(f"nm -D --defined-only {binding.LIB_PATH}").read()
    syms = {line.split()[-1] for line in out.splitlines() if line.strip()}
    ours = {s for s in syms if "grg" in s or s.startswith("lora_")}
    assert ours == set(declared_functions())


def test_workspace_size(lib):
    assert binding.lora_workspace_size(8192, 128) > 0
    assert binding.lora_workspace_size(8192, 128) % 256 == 0
    assert binding.lora_workspace_size(0, 4) == 0
    assert binding.lora_workspace_size(64, 0) == 0
    assert binding.lora_workspace_size(64, binding.LORA_MAX_LORAS + 1) == 0
    assert binding.lora_workspace_size(binding.LORA_MAX_NUM_TOKENS + 1, 4) == 0
    # grows with both sizes, and covers the four tile lists
    small = binding.lora_workspace_size(64, 4)
    assert binding.lora_workspace_size(128, 4) > small
    assert binding.lora_workspace_size(64, 8) > small
    entries = sum((64 + r - 1) // r + 4 for r in (16, 32, 64, 128))
    assert small >= 64 + 8 * entries


def test_shrink_expand_workspace_size(lib):
    base = binding.lora_workspace_size(256, 4)
    # split-K path: up to 16 (rank <= 16) or 8 (rank 32) partial tiles of
    # 16 rows x S*R floats per 16-token tile
    tiles = 256 // 16 + 4
    assert binding.lora_shrink_expand_workspace_size(256, 4, 4096, (4096,) * 3, 8) == \
        base + tiles * 16 * 16 * 24 * 4
    assert binding.lora_shrink_expand_workspace_size(256, 4, 4096, (4096,), 32) == \
        base + tiles * 8 * 16 * 32 * 4
    # beyond 1024 tokens or rank 32 only the metadata part
    assert binding.lora_shrink_expand_workspace_size(2048, 4, 4096, (4096,), 16) == \
        binding.lora_workspace_size(2048, 4)
    assert binding.lora_shrink_expand_workspace_size(256, 4, 4096, (4096,), 64) == base
    # rejected sizes
    assert binding.lora_shrink_expand_workspace_size(256, 4, 4096, (4096,), 12) == 0
    assert binding.lora_shrink_expand_workspace_size(256, 4, 100, (4096,), 8) == 0
    assert binding.lora_shrink_expand_workspace_size(256, 4, 4096, (4095,), 8) == 0
    assert binding.lora_shrink_expand_workspace_size(0, 4, 4096, (4096,), 8) == 0


def test_error_strings(lib):
    for code in range(0, -7, -1):
        assert lib.lora_error_string(code)
    assert b"unknown" in lib.lora_error_string(-99)


# Fake, never-dereferenced pointer values: validation must reject the call
# before anything reaches the GPU.
P16 = 0x10000      # 16-byte aligned
PODD = 0x10002     # misaligned


def _arr(*vals):
    return (ctypes.c_void_p * len(vals))(*vals)


def test_prepare_metadata_validation(lib):
    f = lib.lora_prepare_metadata
    assert f(None, P16, 64, 4, P16, P16, P16, P16, 1 << 20, None) == -1
    assert f(P16, P16, 0, 4, P16, P16, P16, P16, 1 << 20, None) == -3
    assert f(P16, P16, 64, 0, P16, P16, P16, P16, 1 << 20, None) == -3
    assert f(P16, P16, 64, 4, P16, P16, P16, PODD, 1 << 20, None) == -2
    assert f(P16, P16, 64, 4, P16, P16, P16, P16, 16, None) == -4


def test_shrink_validation(lib):
    f = lib.lora_shrink
    a = _arr(P16)
    ws = 1 << 20
    args = dict(x=P16, stride=512, hidden=512, a=ctypes.addressof(a), s=1, r=8, scale=1.0,
                u=P16, sorted=P16, starts=P16, T=64, L=4, ws=P16, wsb=ws)

    def call(**kw):
        d = dict(args, **kw)
        return f(d["x"], d["stride"], d["hidden"], d["a"], d["s"], d["r"], d["scale"], None, d["u"],
                 d["sorted"], d["starts"], d["T"], d["L"], d["ws"], d["wsb"], None)

    assert call(x=None) == -1
    assert call(a=None) == -1
    assert call(a=ctypes.addressof(_arr(None))) == -1
    assert call(s=0) == -3 and call(s=4) == -3
    assert call(r=12) == -3 and call(r=256) == -3
    assert call(hidden=500, stride=504) == -3
    assert call(stride=256) == -3
    assert call(x=PODD) == -2
    assert call(stride=514) == -2
    assert call(u=PODD) == -2
    assert call(a=ctypes.addressof(_arr(PODD))) == -2
    assert call(wsb=8) == -4


def test_expand_validation(lib):
    f = lib.lora_expand
    b = _arr(P16, P16)
    w = (ctypes.c_int64 * 2)(512, 512)

    def call(u=P16, bp=None, wp=None, s=2, r=16, y=P16, ystride=1024, T=64, L=4, ws=P16,
             wsb=1 << 20):
        return f(u, ctypes.addressof(b) if bp is None else bp,
                 ctypes.addressof(w) if wp is None else wp, s, r, y, ystride, P16, P16, T, L, ws,
                 wsb, None)

    assert call(u=None) == -1
    assert call(y=None) == -1
    assert call(wp=0) == -1
    assert call(s=0) == -3
    assert call(r=7) == -3
    assert call(ystride=1000) == -3
    assert call(ystride=1028) == -2
    assert call(y=PODD) == -2
    bad_w = (ctypes.c_int64 * 2)(512, 500)
    assert call(wp=ctypes.addressof(bad_w)) == -3
    assert call(wsb=8) == -4


def test_split_halves_validation(lib):
    """Every call here is rejected before anything is enqueued."""
    big = binding.lora_shrink_expand_workspace_size(64, 4, 512, (512,), 8)
    small = binding.lora_workspace_size(64, 4)
    assert big > small
    a = _arr(P16)
    fs = lib.lora_shrink_partials

    def shrink(x=P16, stride=512, hidden=512, s=1, r=8, T=64, L=4, wsb=big):
        return fs(x, stride, hidden, ctypes.addressof(a), s, r, P16, P16, T, L, P16, wsb, None)

    assert shrink(x=None) == -1
    assert shrink(x=PODD) == -2
    assert shrink(r=12) == -3
    assert shrink(r=64) == -3           # split-K path: rank <= 32
    assert shrink(T=2048, wsb=1 << 24) == -3  # split-K path: up to 1024 tokens
    assert shrink(wsb=small) == -4      # no room for the partial tiles
    b = _arr(P16)
    w = (ctypes.c_int64 * 1)(512)
    fe = lib.lora_expand_partials

    def expand(hidden=512, r=8, u=P16, y=P16, T=64, wsb=big):
        return fe(hidden, ctypes.addressof(b), ctypes.addressof(w), 1, r, 1.0, None, u, y, 512, P16,
                  P16, T, 4, P16, wsb, None)

    assert expand(u=None) == -1
    assert expand(y=PODD) == -2
    assert expand(hidden=500) == -3
    assert expand(r=64) == -3
    assert expand(T=2048, wsb=1 << 24) == -3
    assert expand(wsb=small) == -4


def test_read_status_validation(lib):
    st = ctypes.c_uint32(0)
    assert lib.lora_read_status(None, ctypes.byref(st), None) == -1
    assert lib.lora_read_status(P16, None, None) == -1
    assert lib.lora_read_status(PODD, ctypes.byref(st), None) == -2


def test_binding_refuses_cpu_tensors(lib):
    torch = pytest.importorskip("torch")
    x = torch.zeros(4, 8, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.lora_prepare_metadata(x[0], x[0, :1], 4, x[0], x[0], x[0], x[0])


def test_binding_selects_the_input_type_and_rejects_mixtures():
    torch = pytest.importorskip("torch")
    bf, hf = torch.zeros(2, dtype=torch.bfloat16), torch.zeros(2, dtype=torch.float16)
    assert binding._is_f16([bf, bf]) is False
    assert binding._is_f16([hf, hf]) is True
    with pytest.raises(ValueError):
        binding._is_f16([bf, hf])
    with pytest.raises(ValueError):
        binding._is_f16([torch.zeros(2)])
    with pytest.raises(ValueError):   # entry points without an fp16 variant
        binding._is_f16([hf], fp16_ok=False)


def test_timeout_hook_is_off_by_default_and_reports_its_setting(lib):
    """The test hook of gathered_rank_gemm_testing.h only flips a host flag."""
    assert binding.lora_testing_inject_timeout(False) is False
    assert binding.lora_testing_inject_timeout(True) is False
    assert binding.lora_testing_inject_timeout(False) is True
