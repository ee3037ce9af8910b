"""Thin ctypes binding of the C ABI in ``include/gathered_rank_gemm.h``.

Argument marshalling only: every step of the path runs in the CUDA kernels
of ``libgathered_rank_gemm.so``.  There is no CPU fallback: when the library
is missing or a tensor is not on a CUDA device, the call raises.

PyTorch provides device memory and streams.  Tensors are passed as raw
pointers; the 16-bit operands (x, A, B, y) are all ``torch.bfloat16`` or, with
stacked weights, all ``torch.float16`` (which selects the ``*_f16`` entry
points); the work is
enqueued on ``stream`` (default: the current torch stream of the tensors'
device).
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgathered_rank_gemm.so")

LORA_OK = 0
LORA_STATUS_BAD_LORA_ID = 0x1
LORA_STATUS_BAD_NUM_TOKENS = 0x2
LORA_STATUS_TIMEOUT = 0x4
LORA_STATUS_BAD_WEIGHT = 0x8
LORA_MAX_SLICES = 3
LORA_MAX_LORAS = 1024
LORA_MAX_NUM_TOKENS = 1 << 22

LORA_NOALLOC_SCRATCH_BYTES = 384 * 1024

EXPORTED = ("lora_workspace_size", "lora_prepare_metadata", "lora_shrink", "lora_expand",
            "lora_read_status", "lora_error_string", "lora_apply_noalloc",
            "lora_shrink_expand", "lora_shrink_expand_kernels",
            "lora_shrink_expand_workspace_size", "lora_shrink_partials", "lora_expand_partials",
            "lora_shrink_paged", "lora_expand_paged", "lora_shrink_expand_paged",
            "lora_shrink_f16", "lora_expand_f16", "lora_shrink_expand_f16",
            "lora_shrink_partials_f16", "lora_expand_partials_f16", "lora_shrink_expand_path",
            "lora_testing_inject_timeout")

LORA_PATH_FUSED = 1
LORA_PATH_SPLIT_PAIR = 3
LORA_PATH_PAIR = 4
PATH_NAMES = {LORA_PATH_FUSED: "fused", LORA_PATH_SPLIT_PAIR: "split-K",
              LORA_PATH_PAIR: "cluster"}

_lib = None


class LoraError(RuntimeError):
    """A C-ABI call returned a negative LORA_ERR_* code."""

    def __init__(self, name: str, code: int, text: str):
        super().__init__(f"{name} failed with {code}: {text}")
        self.code = code


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library (built by ``gathered_rank_gemm_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library {path} is missing; build it with "
                           "gathered_rank_gemm_gb300.build.build() (nvcc, sm_103a)")
    lib = ctypes.CDLL(path)
    i64, i32, p, sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
    lib.lora_workspace_size.restype = sz
    lib.lora_workspace_size.argtypes = [i64, i64]
    lib.lora_prepare_metadata.restype = i32
    lib.lora_prepare_metadata.argtypes = [p, p, i64, i64, p, p, p, p, sz, p]
    lib.lora_shrink.restype = i32
    lib.lora_shrink.argtypes = [p, i64, i64, p, i32, i32, ctypes.c_float, p, p, p, p, i64, i64,
                                p, sz, p]
    lib.lora_expand.restype = i32
    lib.lora_expand.argtypes = [p, p, p, i32, i32, p, i64, p, p, i64, i64, p, sz, p]
    lib.lora_read_status.restype = i32
    lib.lora_read_status.argtypes = [p, ctypes.POINTER(ctypes.c_uint32), p]
    lib.lora_error_string.restype = ctypes.c_char_p
    lib.lora_error_string.argtypes = [i32]
    lib.lora_shrink_expand.restype = i32
    lib.lora_shrink_expand.argtypes = [p, i64, i64, p, p, p, i32, i32, ctypes.c_float, p, p, p,
                                       i64, p, p, i64, i64, p, sz, p]
    lib.lora_shrink_expand_kernels.restype = i32
    lib.lora_shrink_expand_kernels.argtypes = [i64, i64, i64, p, i32, i32]
    lib.lora_shrink_expand_workspace_size.restype = sz
    lib.lora_shrink_expand_workspace_size.argtypes = [i64, i64, i64, p, i32, i32]
    lib.lora_shrink_partials.restype = i32
    lib.lora_shrink_partials.argtypes = [p, i64, i64, p, i32, i32, p, p, i64, i64, p, sz, p]
    lib.lora_expand_partials.restype = i32
    lib.lora_expand_partials.argtypes = [i64, p, p, i32, i32, ctypes.c_float, p, p, p, i64, p,
                                         p, i64, i64, p, sz, p]
    lib.lora_shrink_paged.restype = i32
    lib.lora_shrink_paged.argtypes = [p, i64, i64, p, i32, i32, ctypes.c_float, p, p, p, p, i64,
                                      i64, p, sz, p]
    lib.lora_expand_paged.restype = i32
    lib.lora_expand_paged.argtypes = [p, p, p, i32, i32, p, i64, p, p, i64, i64, p, sz, p]
    lib.lora_shrink_expand_paged.restype = i32
    lib.lora_shrink_expand_paged.argtypes = [p, i64, i64, p, p, p, i32, i32, ctypes.c_float, p,
                                             p, p, i64, p, p, i64, i64, p, sz, p]
    for name in ("lora_shrink", "lora_expand", "lora_shrink_expand", "lora_shrink_partials",
                 "lora_expand_partials"):
        f16 = getattr(lib, name + "_f16")
        f16.restype = i32
        f16.argtypes = getattr(lib, name).argtypes
    lib.lora_shrink_expand_path.restype = i32
    lib.lora_shrink_expand_path.argtypes = [i64, i64, i64, p, i32, i32, sz, i32, i32]
    lib.lora_testing_inject_timeout.restype = i32
    lib.lora_testing_inject_timeout.argtypes = [i32]
    lib.lora_apply_noalloc.restype = i32
    lib.lora_apply_noalloc.argtypes = [p, p, i64, i64, p, i64, i64, p, p, p, i32, i32,
                                       ctypes.c_float, p, p, p, i64, p, p, p, p, p]
    _lib = lib
    return lib


def _on_tensor_device(fn):
    """Runs a C-ABI call with the device of its first CUDA tensor argument
    current: the library launches on, and looks its per-device state up for,
    the current device."""
    import functools

    @functools.wraps(fn)
    def wrapped(*args, **kwargs):
        import torch
        for a in list(args) + list(kwargs.values()):
            t = a[0] if isinstance(a, (list, tuple)) and a else a
            if isinstance(t, torch.Tensor) and t.is_cuda:
                with torch.cuda.device(t.device):
                    return fn(*args, **kwargs)
        return fn(*args, **kwargs)
    return wrapped


def _check(name: str, rc: int) -> None:
    if rc != LORA_OK:
        raise LoraError(name, rc, load().lora_error_string(rc).decode())


def _stream_ptr(stream, device) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    return t.data_ptr()


def _scales(lora_scales, num_loras):
    """Device pointer of the per-adapter factors (fp32 [max_loras]) or None."""
    if lora_scales is None:
        return None
    import torch
    if lora_scales.dtype != torch.float32 or lora_scales.numel() != num_loras:
        raise ValueError("lora_scales must be a float32 CUDA tensor of max_loras entries")
    if not lora_scales.is_contiguous():
        raise ValueError("lora_scales must be contiguous")
    return _dev(lora_scales, "lora_scales")


def _is_f16(tensors, fp16_ok=True) -> bool:
    """True for an all-fp16 operand set, False for all-bf16; raises otherwise."""
    import torch
    kinds = {t.dtype for t in tensors}
    if kinds == {torch.bfloat16}:
        return False
    if kinds == {torch.float16} and fp16_ok:
        return True
    allowed = "all bfloat16 or all float16" if fp16_ok else "bfloat16"
    raise ValueError(f"16-bit operands must be {allowed}, got {sorted(map(str, kinds))}")


def _ptr_array(tensors, name):
    arr = (ctypes.c_void_p * len(tensors))(*[_dev(t, f"{name}[{i}]") for i, t in enumerate(tensors)])
    return arr


# ------------------------------------------------------------------ C-ABI calls

def lora_workspace_size(max_num_tokens: int, max_loras: int) -> int:
    return int(load().lora_workspace_size(int(max_num_tokens), int(max_loras)))


@_on_tensor_device
def lora_prepare_metadata(token_lora_mapping, num_tokens, max_loras: int, sorted_token_ids,
                          num_tokens_per_lora, lora_token_start_loc, workspace, stream=None):
    """Stable grouping of the tokens by LoRA id (see the C header)."""
    t_max = token_lora_mapping.shape[0]
    rc = load().lora_prepare_metadata(
        _dev(token_lora_mapping, "token_lora_mapping"), _dev(num_tokens, "num_tokens"), t_max,
        int(max_loras), _dev(sorted_token_ids, "sorted_token_ids"),
        _dev(num_tokens_per_lora, "num_tokens_per_lora"),
        _dev(lora_token_start_loc, "lora_token_start_loc"), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _stream_ptr(stream, workspace.device))
    _check("lora_prepare_metadata", rc)


@_on_tensor_device
def lora_shrink(x, lora_a, scale: float, u, sorted_token_ids, lora_token_start_loc, workspace,
                stream=None, lora_scales=None):
    """u[s][t][r] = scale (* lora_scales[m[t]]) * x[t] . A_s[m[t]][r] for the adapter tokens."""
    lora_a = list(lora_a)
    arr = _ptr_array(lora_a, "lora_a")
    num_loras, rank, hidden = lora_a[0].shape
    fn = load().lora_shrink_f16 if _is_f16([x] + lora_a) else load().lora_shrink
    rc = fn(
        _dev(x, "x"), x.stride(0), hidden, ctypes.addressof(arr), len(lora_a), rank,
        float(scale), _scales(lora_scales, num_loras), _dev(u, "u"), _dev(sorted_token_ids, "sorted_token_ids"),
        _dev(lora_token_start_loc, "lora_token_start_loc"), x.shape[0], num_loras,
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream_ptr(stream, x.device))
    _check("lora_shrink", rc)


@_on_tensor_device
def lora_expand(u, lora_b, y, sorted_token_ids, lora_token_start_loc, workspace, stream=None):
    """y[t][off_s + j] += u[s][t] . B_s[m[t]][:, j] for the adapter tokens (in place)."""
    lora_b = list(lora_b)
    arr = _ptr_array(lora_b, "lora_b")
    widths = (ctypes.c_int64 * len(lora_b))(*[b.shape[2] for b in lora_b])
    num_loras, rank = lora_b[0].shape[:2]
    fn = load().lora_expand_f16 if _is_f16([y] + lora_b) else load().lora_expand
    rc = fn(
        _dev(u, "u"), ctypes.addressof(arr), ctypes.addressof(widths), len(lora_b), rank,
        _dev(y, "y"), y.stride(0), _dev(sorted_token_ids, "sorted_token_ids"),
        _dev(lora_token_start_loc, "lora_token_start_loc"), y.shape[0], num_loras,
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream_ptr(stream, y.device))
    _check("lora_expand", rc)


@_on_tensor_device
def lora_shrink_expand(x, lora_a, lora_b, scale: float, u, y, sorted_token_ids,
                       lora_token_start_loc, workspace, stream=None, lora_scales=None):
    """Shrink then expand in one call (one fused kernel for decode-sized batches)."""
    lora_a, lora_b = list(lora_a), list(lora_b)
    arr_a = _ptr_array(lora_a, "lora_a")
    arr_b = _ptr_array(lora_b, "lora_b")
    widths = (ctypes.c_int64 * len(lora_b))(*[b.shape[2] for b in lora_b])
    num_loras, rank, hidden = lora_a[0].shape
    f16 = _is_f16([x, y] + lora_a + lora_b)
    fn = load().lora_shrink_expand_f16 if f16 else load().lora_shrink_expand
    rc = fn(
        _dev(x, "x"), x.stride(0), hidden, ctypes.addressof(arr_a), ctypes.addressof(arr_b),
        ctypes.addressof(widths), len(lora_a), rank, float(scale),
        _scales(lora_scales, num_loras), _dev(u, "u"), _dev(y, "y"),
        y.stride(0), _dev(sorted_token_ids, "sorted_token_ids"),
        _dev(lora_token_start_loc, "lora_token_start_loc"), x.shape[0], num_loras,
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream_ptr(stream, x.device))
    _check("lora_shrink_expand", rc)


@_on_tensor_device
def lora_shrink_partials(x, lora_a, sorted_token_ids, lora_token_start_loc, workspace,
                         stream=None):
    """Split-K shrink: each CTA's partial tile of u into the workspace (u is not written)."""
    lora_a = list(lora_a)
    arr = _ptr_array(lora_a, "lora_a")
    num_loras, rank, hidden = lora_a[0].shape
    fn = load().lora_shrink_partials_f16 if _is_f16([x] + lora_a) else load().lora_shrink_partials
    rc = fn(
        _dev(x, "x"), x.stride(0), hidden, ctypes.addressof(arr), len(lora_a), rank,
        _dev(sorted_token_ids, "sorted_token_ids"),
        _dev(lora_token_start_loc, "lora_token_start_loc"), x.shape[0], num_loras,
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream_ptr(stream, x.device))
    _check("lora_shrink_partials", rc)


@_on_tensor_device
def lora_expand_partials(hidden: int, lora_b, scale: float, u, y, sorted_token_ids,
                         lora_token_start_loc, workspace, stream=None, lora_scales=None):
    """Sums the split-K partials (scaled) into u, then y += u . B_s (in place)."""
    lora_b = list(lora_b)
    arr = _ptr_array(lora_b, "lora_b")
    widths = (ctypes.c_int64 * len(lora_b))(*[b.shape[2] for b in lora_b])
    num_loras, rank = lora_b[0].shape[:2]
    fn = load().lora_expand_partials_f16 if _is_f16([y] + lora_b) else load().lora_expand_partials
    rc = fn(
        int(hidden), ctypes.addressof(arr), ctypes.addressof(widths), len(lora_b), rank,
        float(scale), _scales(lora_scales, num_loras), _dev(u, "u"), _dev(y, "y"), y.stride(0),
        _dev(sorted_token_ids, "sorted_token_ids"),
        _dev(lora_token_start_loc, "lora_token_start_loc"), y.shape[0], num_loras,
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream_ptr(stream, y.device))
    _check("lora_expand_partials", rc)


def _table_array(tables, name):
    """Host array of the slices' device tables (int64 CUDA tensors of max_loras
    weight addresses; 0 = an all-zero adapter)."""
    import torch
    for i, t in enumerate(tables):
        if t.dtype != torch.int64 or t.dim() != 1 or not t.is_contiguous():
            raise ValueError(f"{name}[{i}] must be a contiguous int64 CUDA tensor of max_loras entries")
    return _ptr_array(tables, name)


@_on_tensor_device
def lora_shrink_paged(x, a_tables, rank: int, scale: float, u, sorted_token_ids,
                      lora_token_start_loc, workspace, stream=None, lora_scales=None):
    """lora_shrink with paged adapter weights: a_tables[s][l] = address of A_s[l] ([rank][hidden])."""
    a_tables = list(a_tables)
    arr = _table_array(a_tables, "a_tables")
    num_loras, hidden = a_tables[0].numel(), x.shape[1]
    _is_f16([x], fp16_ok=False)
    rc = load().lora_shrink_paged(
        _dev(x, "x"), x.stride(0), hidden, ctypes.addressof(arr), len(a_tables), int(rank),
        float(scale), _scales(lora_scales, num_loras), _dev(u, "u"),
        _dev(sorted_token_ids, "sorted_token_ids"),
        _dev(lora_token_start_loc, "lora_token_start_loc"), x.shape[0], num_loras,
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream_ptr(stream, x.device))
    _check("lora_shrink_paged", rc)


@_on_tensor_device
def lora_expand_paged(u, b_tables, slice_widths, y, sorted_token_ids, lora_token_start_loc,
                      workspace, stream=None):
    """lora_expand with paged adapter weights: b_tables[s][l] = address of B_s[l] ([rank][N_s])."""
    b_tables = list(b_tables)
    arr = _table_array(b_tables, "b_tables")
    widths = (ctypes.c_int64 * len(b_tables))(*[int(w) for w in slice_widths])
    num_loras, rank = b_tables[0].numel(), u.shape[2]
    _is_f16([y], fp16_ok=False)
    rc = load().lora_expand_paged(
        _dev(u, "u"), ctypes.addressof(arr), ctypes.addressof(widths), len(b_tables), rank,
        _dev(y, "y"), y.stride(0), _dev(sorted_token_ids, "sorted_token_ids"),
        _dev(lora_token_start_loc, "lora_token_start_loc"), y.shape[0], num_loras,
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream_ptr(stream, y.device))
    _check("lora_expand_paged", rc)


@_on_tensor_device
def lora_shrink_expand_paged(x, a_tables, b_tables, slice_widths, scale: float, u, y,
                             sorted_token_ids, lora_token_start_loc, workspace, stream=None,
                             lora_scales=None):
    """lora_shrink_expand with paged adapter weights."""
    a_tables, b_tables = list(a_tables), list(b_tables)
    arr_a = _table_array(a_tables, "a_tables")
    arr_b = _table_array(b_tables, "b_tables")
    widths = (ctypes.c_int64 * len(b_tables))(*[int(w) for w in slice_widths])
    num_loras, hidden, rank = a_tables[0].numel(), x.shape[1], u.shape[2]
    _is_f16([x, y], fp16_ok=False)
    rc = load().lora_shrink_expand_paged(
        _dev(x, "x"), x.stride(0), hidden, ctypes.addressof(arr_a), ctypes.addressof(arr_b),
        ctypes.addressof(widths), len(a_tables), rank, float(scale),
        _scales(lora_scales, num_loras), _dev(u, "u"), _dev(y, "y"), y.stride(0),
        _dev(sorted_token_ids, "sorted_token_ids"),
        _dev(lora_token_start_loc, "lora_token_start_loc"), x.shape[0], num_loras,
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream_ptr(stream, x.device))
    _check("lora_shrink_expand_paged", rc)


def lora_shrink_expand_kernels(max_num_tokens: int, max_loras: int, hidden: int, slice_widths,
                               rank: int) -> int:
    """Kernels lora_shrink_expand launches for a shape (1 fused, 2 separate)."""
    w = (ctypes.c_int64 * len(slice_widths))(*[int(v) for v in slice_widths])
    rc = load().lora_shrink_expand_kernels(int(max_num_tokens), int(max_loras), int(hidden),
                                           ctypes.addressof(w), len(slice_widths), int(rank))
    if rc < 0:
        _check("lora_shrink_expand_kernels", rc)
    return int(rc)


def lora_shrink_expand_path(max_num_tokens: int, max_loras: int, hidden: int, slice_widths,
                            rank: int, workspace_bytes: int, fp16: bool = False,
                            paged: bool = False) -> int:
    """Which path one lora_shrink_expand call takes (LORA_PATH_*) for a shape
    and workspace size on the current device."""
    w = (ctypes.c_int64 * len(slice_widths))(*[int(v) for v in slice_widths])
    rc = load().lora_shrink_expand_path(int(max_num_tokens), int(max_loras), int(hidden),
                                        ctypes.addressof(w), len(slice_widths), int(rank),
                                        int(workspace_bytes), int(bool(fp16)), int(bool(paged)))
    if rc < 0:
        _check("lora_shrink_expand_path", rc)
    return int(rc)


def lora_shrink_expand_workspace_size(max_num_tokens: int, max_loras: int, hidden: int,
                                      slice_widths, rank: int) -> int:
    """Workspace bytes that let lora_shrink_expand take its split-K path."""
    w = (ctypes.c_int64 * len(slice_widths))(*[int(v) for v in slice_widths])
    return int(load().lora_shrink_expand_workspace_size(
        int(max_num_tokens), int(max_loras), int(hidden), ctypes.addressof(w),
        len(slice_widths), int(rank)))


@_on_tensor_device
def lora_read_status(workspace, stream=None) -> int:
    """Status bits OR-ed since the last read (synchronises the stream, clears them)."""
    out = ctypes.c_uint32(0)
    rc = load().lora_read_status(_dev(workspace, "workspace"), ctypes.byref(out),
                                 _stream_ptr(stream, workspace.device))
    _check("lora_read_status", rc)
    return int(out.value)


def lora_testing_inject_timeout(on: bool) -> bool:
    """Test hook (include/gathered_rank_gemm_testing.h): while on, the shrink
    kernel's bounded waits run out after 1 ms and it reports
    LORA_STATUS_TIMEOUT.  Returns the previous setting."""
    return bool(load().lora_testing_inject_timeout(1 if on else 0))


@_on_tensor_device
def lora_apply_noalloc(token_lora_mapping, num_tokens, x, lora_a, lora_b, scale: float, u, y,
                       sorted_token_ids, num_tokens_per_lora, lora_token_start_loc,
                       status=None, stream=None, lora_scales=None):
    """Grouping + shrink + expand of one layer without any allocation.

    For callers that cannot allocate device memory: the workspace is the
    library's static device array (LORA_NOALLOC_SCRATCH_BYTES), shared by all
    calls, so calls that overlap on the GPU race.  The first call on a device
    looks the array up; make it before any stream capture.  ``status``: an
    optional int32 CUDA tensor of one element receiving the status bits.
    """
    lora_a, lora_b = list(lora_a), list(lora_b)
    arr_a = _ptr_array(lora_a, "lora_a")
    arr_b = _ptr_array(lora_b, "lora_b")
    widths = (ctypes.c_int64 * len(lora_b))(*[b.shape[2] for b in lora_b])
    num_loras, rank, hidden = lora_a[0].shape
    _is_f16([x, y] + lora_a + lora_b, fp16_ok=False)
    rc = load().lora_apply_noalloc(
        _dev(token_lora_mapping, "token_lora_mapping"), _dev(num_tokens, "num_tokens"),
        token_lora_mapping.shape[0], num_loras, _dev(x, "x"), x.stride(0), hidden,
        ctypes.addressof(arr_a), ctypes.addressof(arr_b), ctypes.addressof(widths), len(lora_a),
        rank, float(scale), _scales(lora_scales, num_loras), _dev(u, "u"), _dev(y, "y"),
        y.stride(0), _dev(sorted_token_ids, "sorted_token_ids"),
        _dev(num_tokens_per_lora, "num_tokens_per_lora"),
        _dev(lora_token_start_loc, "lora_token_start_loc"),
        None if status is None else _dev(status, "status"), _stream_ptr(stream, x.device))
    _check("lora_apply_noalloc", rc)


# ------------------------------------------------------------------ buffers

class LoraMetadata:
    """Device buffers of one batch's grouping (sized by max_num_tokens / max_loras)."""

    def __init__(self, max_num_tokens: int, max_loras: int, device="cuda", workspace_bytes=None):
        """workspace_bytes: None for lora_workspace_size, or a larger size such
        as lora_shrink_expand_workspace_size for the one-call split-K path."""
        import torch
        self.max_num_tokens = int(max_num_tokens)
        self.max_loras = int(max_loras)
        i32 = dict(dtype=torch.int32, device=device)
        self.sorted_token_ids = torch.empty(self.max_num_tokens, **i32)
        self.num_tokens_per_lora = torch.empty(self.max_loras + 1, **i32)
        self.lora_token_start_loc = torch.empty(self.max_loras + 2, **i32)
        base = lora_workspace_size(self.max_num_tokens, self.max_loras)
        if base == 0:
            raise ValueError("max_num_tokens / max_loras outside the supported range")
        nbytes = base if workspace_bytes is None else max(int(workspace_bytes), base)
        self.workspace = torch.zeros(nbytes, dtype=torch.uint8, device=device)

    def prepare(self, token_lora_mapping, num_tokens, stream=None):
        lora_prepare_metadata(token_lora_mapping, num_tokens, self.max_loras,
                              self.sorted_token_ids, self.num_tokens_per_lora,
                              self.lora_token_start_loc, self.workspace, stream)

    def shrink(self, x, lora_a, scale, u, stream=None, lora_scales=None):
        lora_shrink(x, lora_a, scale, u, self.sorted_token_ids, self.lora_token_start_loc,
                    self.workspace, stream, lora_scales)

    def expand(self, u, lora_b, y, stream=None):
        lora_expand(u, lora_b, y, self.sorted_token_ids, self.lora_token_start_loc,
                    self.workspace, stream)

    def shrink_expand(self, x, lora_a, lora_b, scale, u, y, stream=None, lora_scales=None):
        lora_shrink_expand(x, lora_a, lora_b, scale, u, y, self.sorted_token_ids,
                           self.lora_token_start_loc, self.workspace, stream, lora_scales)

    def shrink_partials(self, x, lora_a, stream=None):
        lora_shrink_partials(x, lora_a, self.sorted_token_ids, self.lora_token_start_loc,
                             self.workspace, stream)

    def expand_partials(self, hidden, lora_b, scale, u, y, stream=None, lora_scales=None):
        lora_expand_partials(hidden, lora_b, scale, u, y, self.sorted_token_ids,
                             self.lora_token_start_loc, self.workspace, stream, lora_scales)

    def shrink_paged(self, x, a_tables, rank, scale, u, stream=None, lora_scales=None):
        lora_shrink_paged(x, a_tables, rank, scale, u, self.sorted_token_ids,
                          self.lora_token_start_loc, self.workspace, stream, lora_scales)

    def expand_paged(self, u, b_tables, slice_widths, y, stream=None):
        lora_expand_paged(u, b_tables, slice_widths, y, self.sorted_token_ids,
                          self.lora_token_start_loc, self.workspace, stream)

    def shrink_expand_paged(self, x, a_tables, b_tables, slice_widths, scale, u, y, stream=None,
                            lora_scales=None):
        lora_shrink_expand_paged(x, a_tables, b_tables, slice_widths, scale, u, y,
                                 self.sorted_token_ids, self.lora_token_start_loc,
                                 self.workspace, stream, lora_scales)

    def read_status(self, stream=None) -> int:
        return lora_read_status(self.workspace, stream)
