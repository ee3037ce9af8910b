"""The allocation-free entry point (lora_apply_noalloc) against the regular path.

Some callers cannot allocate device memory, so they cannot hand the library
the workspace that lora_prepare_metadata / lora_shrink / lora_expand take.
lora_apply_noalloc runs the same layer with its workspace in a static device
array of the library.  This file checks, through the C ABI, that two calls in
a row give the same u, y and metadata as the regular entry points (within the
tolerance the other parity tests use), and that sizes beyond the static array
are refused before anything runs.  It is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

from gathered_rank_gemm_gb300 import binding
from gathered_rank_gemm_gb300 import workloads as W

torch = pytest.importorskip("torch")


def _regular(shape, mapping, layer, dev):
    """y, u and metadata from prepare + shrink + expand with their own workspace."""
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    meta = binding.LoraMetadata(shape.max_num_tokens, shape.max_loras, dev)
    m = torch.from_numpy(mapping).to(dev)
    n = torch.tensor([shape.num_tokens], dtype=torch.int32, device=dev)
    y = bf(layer.y)
    u = torch.zeros(shape.num_slices, shape.max_num_tokens, shape.rank, device=dev)
    meta.prepare(m, n)
    meta.shrink(bf(layer.x), [bf(a) for a in layer.lora_a], shape.scale, u)
    meta.expand(u, [bf(b) for b in layer.lora_b], y)
    torch.cuda.synchronize()
    return y.float(), u, meta


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["decode_qkv", "ragged", "down_proj_graph"])
def test_noalloc_matches_the_regular_path_twice(name):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gathered_rank_gemm_gb300 import build
    build.build()
    binding.load()
    dev = torch.device("cuda:0")
    if name == "ragged":
        shape = W.custom_shape(max_num_tokens=300, num_tokens=211, hidden=520,
                               slice_widths=(264, 72), max_loras=6, rank=16, neg_prob=0.2)
    else:
        shape = W.CONFIGS[name]
    rng = np.random.default_rng(77)
    mapping = W.make_mapping(shape, rng)
    layer = W.make_layer(shape, rng)
    y_ref, u_ref, meta = _regular(shape, mapping, layer, dev)
    rows = np.nonzero((mapping[:shape.num_tokens] >= 0) &
                      (mapping[:shape.num_tokens] < shape.max_loras))[0]
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    x = bf(layer.x)
    a = [bf(v) for v in layer.lora_a]
    b = [bf(v) for v in layer.lora_b]
    m = torch.from_numpy(mapping).to(dev)
    n = torch.tensor([shape.num_tokens], dtype=torch.int32, device=dev)
    for call in range(2):   # the static array keeps the previous call's contents
        y = bf(layer.y)
        u = torch.zeros(shape.num_slices, shape.max_num_tokens, shape.rank, device=dev)
        sorted_ids = torch.full((shape.max_num_tokens,), 7, dtype=torch.int32, device=dev)
        counts = torch.full((shape.max_loras + 1,), 7, dtype=torch.int32, device=dev)
        starts = torch.full((shape.max_loras + 2,), 7, dtype=torch.int32, device=dev)
        status = torch.full((1,), 99, dtype=torch.int32, device=dev)
        binding.lora_apply_noalloc(m, n, x, a, b, shape.scale, u, y, sorted_ids, counts, starts,
                                   status)
        torch.cuda.synchronize()
        assert torch.equal(sorted_ids, meta.sorted_token_ids)
        assert torch.equal(counts, meta.num_tokens_per_lora)
        assert torch.equal(starts, meta.lora_token_start_loc)
        assert status.item() == 0
        yr = y_ref[rows]
        assert torch.all((y.float()[rows] - yr).abs() <= 1e-2 + 1e-2 * yr.abs()), call
        ur = u_ref[:, rows]
        assert torch.all((u[:, rows] - ur).abs() <= 1e-2 + 1e-2 * ur.abs()), call
        # rows without an adapter keep the input exactly
        keep = np.setdiff1d(np.arange(shape.max_num_tokens), rows)
        assert torch.equal(y[keep].view(torch.int16), bf(layer.y)[keep].view(torch.int16))


def test_noalloc_refuses_sizes_beyond_the_static_array():
    # validation runs before anything touches the GPU, so fake pointers are safe
    from gathered_rank_gemm_gb300 import build
    build.build()
    lib = binding.load()
    big_t, big_l = 1 << 20, 1024
    assert binding.lora_workspace_size(big_t, big_l) > binding.LORA_NOALLOC_SCRATCH_BYTES
    P = 0x10000
    arr = (ctypes.c_void_p * 1)(P)
    w = (ctypes.c_int64 * 1)(64)
    rc = lib.lora_apply_noalloc(P, P, big_t, big_l, P, 64, 64, ctypes.addressof(arr),
                                ctypes.addressof(arr), ctypes.addressof(w), 1, 8, 1.0, None, P,
                                P, 64, P, P, P, None, None)
    assert rc == -4   # LORA_ERR_WORKSPACE
    assert binding.lora_workspace_size(8192, 128) <= binding.LORA_NOALLOC_SCRATCH_BYTES
