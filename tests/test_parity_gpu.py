"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Metadata is compared bit-exactly over whole buffers; u and y per element
within |gpu - oracle| <= 1e-2 + 1e-2 |oracle|; rows without an adapter, pad
rows, columns past the slices and guard bands bit-exactly against their
pre-call contents.
"""
import numpy as np
import pytest

import oracle
from gathered_rank_gemm_gb300 import binding
from gathered_rank_gemm_gb300 import workloads as W

from helpers import (DeviceCase, U_SENTINEL_BITS, bf16_dev, bits_of, check_case, lora_rows,
                     within_tol)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gathered_rank_gemm_gb300 import build
    build.build()
    binding.load()
    return torch.device("cuda:0")


def make_case(shape, dev, seed=0, **kw):
    rng = np.random.default_rng(seed)
    mapping = W.make_mapping(shape, rng)
    layer = W.make_layer(shape, rng)
    return DeviceCase(shape, mapping, layer, dev, **kw)


# ------------------------------------------------------------ the five workloads

@pytest.mark.parametrize("name", ["tiny", "decode_qkv", "chunked_prefill", "mlp_gate_up",
                                  "down_proj_graph"])
def test_named_workload_full_size(name, dev):
    wl = W.make_workload(name)
    case = DeviceCase(wl.shape, wl.mapping, wl.layers[0], dev)
    info = check_case(case)   # every adapter row
    assert case.ws.view[:4].view(torch.int32).item() == 0   # status clean
    print(name, info)


# ------------------------------------------------------------ shapes and ragged edges

SHAPES = [
    # (T, n, H, widths, L, R, mapping)
    (48, 48, 520, (264,), 3, 8, "uniform"),            # H not a multiple of 64, width not of 256
    (100, 77, 136, (40, 24, 16), 5, 16, "uniform"),    # three unequal slices, pad rows
    (300, 300, 1000, (72, 200), 7, 32, "zipf"),        # rank 32, two slices
    (130, 129, 256, (128,), 2, 64, "uniform"),         # rank 64
    (70, 70, 384, (96, 96, 96), 3, 128, "uniform"),    # rank 128, three slices (S*R = 384)
    (64, 64, 64, (8,), 1, 8, "uniform"),               # one LoRA, narrowest slice
    (1, 1, 8, (8,), 1, 8, "all_zero"),                 # a single token, smallest sizes
    (2048, 1500, 512, (512,), 16, 16, "runs"),         # long runs, pad rows
]


@pytest.mark.parametrize("T,n,H,widths,L,R,kind", SHAPES)
def test_ragged_and_edge_shapes(T, n, H, widths, L, R, kind, dev):
    shape = W.custom_shape(max_num_tokens=T, num_tokens=n, hidden=H, slice_widths=widths,
                           max_loras=L, rank=R, mapping=kind, neg_prob=0.15)
    case = make_case(shape, dev, seed=T + H + R)
    check_case(case)


# 32-token tiles of narrow adapters (S*R <= 32) over at least 32 k-blocks:
# the shrink's stages hold four k-blocks each, in lora_shrink and in the one
# call (whose expand then starts at the shrink's end).  A short last group
# and a last k-block past the hidden size (2120, 3000), run tiles (one TMA box
# per k-block) and gathered tiles, one to three slices.
KGROUP_SHAPES = [
    (2048, 2000, 2120, (264,), 6, 16, "runs"),
    (4096, 3900, 4096, (512, 520), 8, 16, "runs"),
    (1100, 1100, 2048, (256, 128, 136), 5, 8, "uniform"),
    (1500, 1400, 3000, (1024,), 3, 32, "runs"),
    # one column tile (S*R = 8) in the two-tile kernel
    (1536, 1500, 2048, (512,), 4, 8, "runs"),
    # 24 k-blocks over clusters of two (enough tiles for three CTAs per SM):
    # twelve one-k-block stages per CTA in the two-tile kernel, S*R = 16 and 8
    (8192, 8000, 1536, (512,), 8, 16, "runs"),
    (8192, 7900, 1536, (256,), 6, 8, "uniform"),
]


@pytest.mark.parametrize("one_call", [False, True])
@pytest.mark.parametrize("T,n,H,widths,L,R,kind", KGROUP_SHAPES)
def test_k_group_stages_match_the_oracle(T, n, H, widths, L, R, kind, one_call, dev):
    shape = W.custom_shape(max_num_tokens=T, num_tokens=n, hidden=H, slice_widths=widths,
                           max_loras=L, rank=R, mapping=kind, neg_prob=0.1)
    check_case(make_case(shape, dev, seed=T + H + R), fused=one_call)


@pytest.mark.parametrize("R", [8, 16, 32, 64, 128])
@pytest.mark.parametrize("S", [1, 2, 3])
def test_every_rank_and_slice_count(R, S, dev):
    shape = W.custom_shape(max_num_tokens=96, num_tokens=90, hidden=192, slice_widths=(64,) * S,
                           max_loras=4, rank=R, mapping="uniform", neg_prob=0.1)
    check_case(make_case(shape, dev, seed=R * 10 + S))


def test_strided_rows_are_respected(dev):
    shape = W.custom_shape(max_num_tokens=80, num_tokens=80, hidden=256, slice_widths=(128, 64),
                           max_loras=3, rank=16)
    case = make_case(shape, dev, seed=3, x_pad=40, y_pad=24)
    check_case(case)


@pytest.mark.parametrize("one_call", [False, True])
def test_strided_rows_on_run_tiles_and_k_group_stages(one_call, dev):
    """Padded x and y rows where the shrink loads run tiles as TMA boxes of a
    tensor map over x (its row stride is the caller's), in stages of four
    k-blocks for lora_shrink and of one in the one call (hidden 2112: a
    short last group)."""
    shape = W.custom_shape(max_num_tokens=2048, num_tokens=2000, hidden=2112,
                           slice_widths=(264,), max_loras=6, rank=16, mapping="runs",
                           neg_prob=0.05)
    case = make_case(shape, dev, seed=7, x_pad=40, y_pad=24)
    check_case(case, fused=one_call)


def test_no_tokens_changes_nothing(dev):
    shape = W.custom_shape(max_num_tokens=64, num_tokens=0, hidden=128, slice_widths=(64,),
                           max_loras=2, rank=8)
    case = make_case(shape, dev)
    check_case(case)
    assert np.all(case.sorted.view.cpu().numpy() == -1)


def test_all_tokens_without_adapter(dev):
    shape = W.custom_shape(max_num_tokens=64, num_tokens=64, hidden=128, slice_widths=(64,),
                           max_loras=2, rank=8, neg_prob=1.0)
    check_case(make_case(shape, dev))


def test_long_batch_takes_several_register_chunks(dev):
    # more than 32 warps x 512 tokens: the grouping reloads the mapping per chunk
    shape = W.custom_shape(max_num_tokens=40000, num_tokens=39000, hidden=64, slice_widths=(64,),
                           max_loras=7, rank=8, mapping="runs", neg_prob=0.0)
    check_case(make_case(shape, dev, seed=40))


def test_many_loras_uses_every_bin(dev):
    shape = W.custom_shape(max_num_tokens=4096, num_tokens=4096, hidden=64, slice_widths=(64,),
                           max_loras=1024, rank=8, neg_prob=0.05)
    check_case(make_case(shape, dev, seed=9))


# ------------------------------------------------------------ exact integer cases

def _int_case(dev, T, H, sparse_k=None, seed=0, R=8, widths=(16, 8), **kw):
    rng = np.random.default_rng(seed)
    L = 3
    if sparse_k is None:
        xi = rng.choice([-2, 0, 2], size=(T, H))
    else:
        xi = np.zeros((T, H), np.int64)
        for t in range(T):
            xi[t, rng.choice(H, sparse_k, replace=False)] = rng.choice([-2, 2], size=sparse_k)
    ai = [rng.choice([-1, 0, 1], size=(L, R, H)) for _ in widths]
    bi = [rng.choice([-1, 0, 1], size=(L, R, w)) for w in widths]
    yi = rng.integers(-8, 9, size=(T, sum(widths)))
    m = rng.integers(-1, L, size=T).astype(np.int32)
    f = lambda a: W.f32_to_bf16_bits(np.asarray(a, np.float32))
    shape = W.custom_shape(max_num_tokens=T, num_tokens=T, hidden=H, slice_widths=widths,
                           max_loras=L, rank=R, scale=0.5)
    layer = W.Layer(x=f(xi), lora_a=[f(v) for v in ai], lora_b=[f(v) for v in bi], y=f(yi))
    return DeviceCase(shape, m, layer, dev, **kw), (xi, ai, bi, yi, m)


INT_PATHS = [
    # (T, H, nonzeros per x row, one call, split-K workspace, expected one-call kernels)
    (24, 16, None, False, False, None),
    (64, 4096, 16, False, False, None),
    (24, 16, None, True, False, 1),       # the fused kernel
    (64, 4096, 16, True, False, 1),       # the fused kernel, a long hidden dimension
    (64, 8200, 16, True, True, 2),        # the split-K pair
    (1100, 1032, 16, True, False, 2),     # the cluster pair (past the split-K sizes)
    (1100, 2120, 16, False, False, None),  # shrink stages of four k-blocks, the last short
    (1100, 2120, 16, True, False, 2),     # the cluster pair on the same shape
]


@pytest.mark.parametrize("T,H,sparse,one_call,split_ws,kernels", INT_PATHS)
def test_small_integer_inputs_are_bit_exact(T, H, sparse, one_call, split_ws, kernels, dev):
    """Every product and partial sum is an integer of modest size, exact in
    fp32 and bf16 whatever the summation order: every path must give the
    oracle's values bit for bit."""
    case, (xi, ai, bi, yi, m) = _int_case(dev, T, H, sparse, seed=H, split_workspace=split_ws)
    if kernels is not None:
        sh = case.shape
        assert binding.lora_shrink_expand_kernels(T, sh.max_loras, H, sh.slice_widths,
                                                  sh.rank) == kernels
    case.run(fused=one_call)
    if split_ws:
        assert torch.any(case.ws.view[case.ws_base:] != 0)   # the split-K path ran
    u = case.u.view.cpu().numpy()
    y = oracle.bf16_bits_to_f64(bits_of(case.y.view))
    u_ref = oracle.shrink(case.layer.x, case.layer.lora_a, 0.5, m, T, 3,
                          u_init=np.zeros((2, T, case.shape.rank)))
    y_ref = oracle.expand(u_ref, case.layer.lora_b, case.layer.y, m, T, 3)
    rows = lora_rows(m, T, 3)
    assert np.array_equal(u[:, rows].astype(np.float64), u_ref[:, rows])
    assert np.array_equal(y, y_ref)


# ------------------------------------------------------------ invariants

def test_one_adapter_batch_equals_dense_fp32_torch(dev):
    T, H, N, R = 200, 1024, 768, 16
    shape = W.custom_shape(max_num_tokens=T, num_tokens=T, hidden=H, slice_widths=(N,),
                           max_loras=2, rank=R, mapping="all_zero", scale=0.75)
    case = make_case(shape, dev, seed=4)
    x32 = case.x.float()
    a32 = case.a[0][0].float()
    b32 = case.b[0][0].float()
    y0 = case.y_view.float().clone()
    case.run()
    u_dense = 0.75 * (x32 @ a32.T)
    y_dense = y0 + u_dense @ b32
    u = case.u.view[0]
    assert torch.all((u - u_dense).abs() <= 1e-2 + 1e-2 * u_dense.abs())
    y = case.y_view.float()
    assert torch.all((y - y_dense).abs() <= 1e-2 + 1e-2 * y_dense.abs())


def test_zero_base_output_isolates_the_delta(dev):
    shape = W.CONFIGS["decode_qkv"]
    wl = W.make_workload(shape)
    layer = wl.layers[0]
    layer = W.Layer(x=layer.x, lora_a=layer.lora_a, lora_b=layer.lora_b,
                    y=np.zeros_like(layer.y))
    case = DeviceCase(shape, wl.mapping, layer, dev)
    case.run()
    rows = lora_rows(wl.mapping, shape.num_tokens, shape.max_loras)
    u_ref = oracle.shrink(layer.x, layer.lora_a, 1.0, wl.mapping, shape.num_tokens, 4,
                          u_init=np.zeros((3, shape.max_num_tokens, 8)))
    d_ref = oracle.expand(u_ref, layer.lora_b, layer.y, wl.mapping, shape.num_tokens, 4)
    d = oracle.bf16_bits_to_f64(bits_of(case.y.view))
    ok, worst = within_tol(d[rows], d_ref[rows])
    assert ok
    # the delta is small (std ~0.07): also hold it to bf16 precision, relative
    rel = np.abs(d[rows] - d_ref[rows]) / (np.abs(d_ref[rows]) + 1e-3)
    assert np.median(rel) < 4e-3


def test_token_permutation_permutes_the_outputs(dev):
    shape = W.custom_shape(max_num_tokens=256, num_tokens=256, hidden=512, slice_widths=(256,),
                           max_loras=4, rank=16)
    rng = np.random.default_rng(17)
    m = W.make_mapping(shape, rng)
    layer = W.make_layer(shape, rng)
    perm = rng.permutation(256)
    c1 = DeviceCase(shape, m, layer, dev)
    c1.run()
    lp = W.Layer(x=layer.x[perm], lora_a=layer.lora_a, lora_b=layer.lora_b, y=layer.y[perm])
    c2 = DeviceCase(shape, np.ascontiguousarray(m[perm]), lp, dev)
    c2.run()
    y1 = c1.y_view.float().cpu().numpy()[perm]
    y2 = c2.y_view.float().cpu().numpy()
    assert np.all(np.abs(y1 - y2) <= 1e-2 + 1e-2 * np.abs(y1))


def test_bad_ids_and_bad_n_set_status_bits(dev):
    shape = W.custom_shape(max_num_tokens=64, num_tokens=64, hidden=64, slice_widths=(64,),
                           max_loras=4, rank=8)
    rng = np.random.default_rng(2)
    m = W.make_mapping(shape, rng)
    m[[3, 17, 40]] = [4, 1000, -5]          # out of range: treated as no adapter
    case = DeviceCase(shape, m, W.make_layer(shape, rng), dev)
    check_case(case)
    assert case.ws.view[:4].view(torch.int32).item() == binding.LORA_STATUS_BAD_LORA_ID
    st = binding.lora_read_status(case.ws.view)
    assert st == binding.LORA_STATUS_BAD_LORA_ID
    assert binding.lora_read_status(case.ws.view) == 0      # cleared by the read
    case.n.fill_(65)                                          # n > max_num_tokens: clamped
    case.prepare()
    assert binding.lora_read_status(case.ws.view) & binding.LORA_STATUS_BAD_NUM_TOKENS
    assert case.starts.view[-1].item() == 64


def test_argument_errors_launch_nothing(dev):
    shape = W.custom_shape(max_num_tokens=64, num_tokens=64, hidden=64, slice_widths=(64,),
                           max_loras=2, rank=8)
    case = make_case(shape, dev)
    case.run()
    y_before = bits_of(case.y.view).copy()
    with pytest.raises(binding.LoraError):
        binding.lora_expand(case.u.view, case.b, case.y_view, case.sorted.view,
                            case.starts.view, case.ws.view[:8])
    with pytest.raises(binding.LoraError):
        binding.lora_shrink(case.x[:, 1:], case.a, 1.0, case.u.view, case.sorted.view,
                            case.starts.view, case.ws.view)
    torch.cuda.synchronize()
    assert np.array_equal(bits_of(case.y.view), y_before)


# ------------------------------------------------------------ CUDA graphs

def test_graph_captured_once_replays_new_mappings_and_n(dev):
    sh = W.custom_shape(max_num_tokens=1024, num_tokens=700, hidden=1024, slice_widths=(512,),
                        max_loras=32, rank=32, neg_prob=0.25)
    if True:
        rng = np.random.default_rng(8)
        m1 = W.make_mapping(sh, rng)
        layer = W.make_layer(sh, rng)
        g_case = DeviceCase(sh, m1, layer, dev)
        stream = torch.cuda.Stream()
        y_clean = g_case.y.view.clone()
        g_case.u.view.view(torch.int32).fill_(U_SENTINEL_BITS)
        torch.cuda.synchronize()
        # warm up on the side stream (sets kernel attributes), then capture
        with torch.cuda.stream(stream):
            g_case.prepare(stream); g_case.shrink(stream); g_case.expand(stream)
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            g_case.prepare(stream)
            g_case.shrink(stream)
            g_case.expand(stream)
        for trial, n_new in enumerate((700, 333, 1024, 0)):
            m_new = W.make_mapping(W.custom_shape(max_num_tokens=1024, num_tokens=n_new,
                                                  hidden=8, slice_widths=(8,), max_loras=32,
                                                  rank=8, neg_prob=0.3),
                                   np.random.default_rng(100 + trial))
            g_case.mapping.copy_(torch.from_numpy(m_new))
            g_case.n.fill_(n_new)
            g_case.y.view.copy_(y_clean)
            g_case.u.view.view(torch.int32).fill_(U_SENTINEL_BITS)
            torch.cuda.synchronize()
            graph.replay()
            torch.cuda.synchronize()
            # a fresh eager run on separate buffers must agree bit for bit
            sh2 = W.custom_shape(max_num_tokens=1024, num_tokens=n_new, hidden=1024,
                                 slice_widths=(512,), max_loras=32, rank=32)
            eager = DeviceCase(sh2, m_new, layer, dev)
            eager.run()
            assert torch.equal(g_case.sorted.view, eager.sorted.view)
            assert torch.equal(g_case.starts.view, eager.starts.view)
            assert torch.equal(g_case.y.view.view(torch.int16), eager.y.view.view(torch.int16))
            assert torch.equal(g_case.u.view.view(torch.int32), eager.u.view.view(torch.int32))


def test_graph_with_run_tiles_and_k_group_stages(dev):
    """lora_shrink's four-k-block stages and run tiles (TMA boxes of x) in a
    graph captured once: replays with new request-run mappings and new n
    equal eager runs on separate buffers bit for bit."""
    T, H, widths, L, R = 2048, 2112, (264,), 6, 16
    sh = W.custom_shape(max_num_tokens=T, num_tokens=T, hidden=H, slice_widths=widths,
                        max_loras=L, rank=R, mapping="runs", neg_prob=0.05)
    rng = np.random.default_rng(21)
    layer = W.make_layer(sh, rng)
    g_case = DeviceCase(sh, W.make_mapping(sh, rng), layer, dev)
    stream = torch.cuda.Stream()
    y_clean = g_case.y.view.clone()
    with torch.cuda.stream(stream):
        g_case.prepare(stream); g_case.shrink(stream); g_case.expand(stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        g_case.prepare(stream)
        g_case.shrink(stream)
        g_case.expand(stream)
    for trial, n_new in enumerate((T, 1500, 1111)):
        m_new = W.make_mapping(W.custom_shape(max_num_tokens=T, num_tokens=n_new, hidden=8,
                                              slice_widths=(8,), max_loras=L, rank=8,
                                              mapping="runs", neg_prob=0.05),
                               np.random.default_rng(200 + trial))
        g_case.mapping.copy_(torch.from_numpy(m_new))
        g_case.n.fill_(n_new)
        g_case.y.view.copy_(y_clean)
        g_case.u.view.view(torch.int32).fill_(U_SENTINEL_BITS)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        sh2 = W.custom_shape(max_num_tokens=T, num_tokens=n_new, hidden=H, slice_widths=widths,
                             max_loras=L, rank=R)
        eager = DeviceCase(sh2, m_new, layer, dev)
        eager.run()
        assert torch.equal(g_case.sorted.view, eager.sorted.view)
        assert torch.equal(g_case.y.view.view(torch.int16), eager.y.view.view(torch.int16))
        assert torch.equal(g_case.u.view.view(torch.int32), eager.u.view.view(torch.int32))


def test_down_proj_workload_inside_a_graph(dev):
    wl = W.make_workload("down_proj_graph")
    sh = wl.shape
    case = DeviceCase(sh, wl.mapping, wl.layers[0], dev)
    stream = torch.cuda.Stream()
    y0 = case.y.view.clone()
    with torch.cuda.stream(stream):
        case.prepare(stream); case.shrink(stream); case.expand(stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        case.prepare(stream); case.shrink(stream); case.expand(stream)
    for _ in range(2):
        case.y.view.copy_(y0)
        case.u.view.view(torch.int32).fill_(U_SENTINEL_BITS)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        rows = lora_rows(wl.mapping, sh.num_tokens, sh.max_loras)
        lay = wl.layers[0]
        if _ == 0:
            u_ref = oracle.shrink(lay.x, lay.lora_a, 1.0, wl.mapping, sh.num_tokens, sh.max_loras,
                                  u_init=np.zeros((1, sh.max_num_tokens, sh.rank)))
            y_ref = oracle.expand(u_ref, lay.lora_b, lay.y, wl.mapping, sh.num_tokens,
                                  sh.max_loras)
        y = oracle.bf16_bits_to_f64(bits_of(case.y.view))
        ok, worst = within_tol(y[rows], y_ref[rows])
        assert ok, worst
        tail = bits_of(case.y.view)[sh.num_tokens:]
        assert np.all(tail == W.BF16_Y_SENTINEL)
        u_bits = case.u.view.cpu().numpy().view(np.uint32)
        assert np.all(u_bits[:, sh.num_tokens:] == U_SENTINEL_BITS)


# ------------------------------------------------------------ one-call shrink + expand

FUSED_SHAPES = [
    ("decode_qkv", None),
    ("tiny", None),
    ("chunked_prefill", None),
    ("mlp_gate_up", None),
    ("down_proj_graph", None),
    ("ragged3", (300, 211, 520, (264, 72, 136), 6, 8)),
    ("rank16", (256, 256, 1024, (512, 512), 4, 16)),
    ("rank32_two_slices", (1500, 1400, 776, (520, 264), 5, 32)),
    ("rank64", (128, 120, 256, (256,), 3, 64)),
    ("rank128_three_slices", (96, 90, 512, (128, 64, 192), 2, 128)),
    ("prefill_like", (4096, 4000, 512, (512,), 8, 16)),
]


@pytest.mark.parametrize("name,spec", FUSED_SHAPES)
def test_shrink_expand_one_call_matches_the_oracle(name, spec, dev):
    if spec is None:
        wl = W.make_workload(name)
        case = DeviceCase(wl.shape, wl.mapping, wl.layers[0], dev)
    else:
        T, n, H, widths, L, R = spec
        shape = W.custom_shape(max_num_tokens=T, num_tokens=n, hidden=H, slice_widths=widths,
                               max_loras=L, rank=R, neg_prob=0.15)
        case = make_case(shape, dev, seed=T + R)
    check_case(case, fused=True)   # every adapter row


def test_shrink_expand_one_call_equals_the_two_calls(dev):
    wl = W.make_workload("decode_qkv")
    a = DeviceCase(wl.shape, wl.mapping, wl.layers[0], dev)
    b = DeviceCase(wl.shape, wl.mapping, wl.layers[0], dev)
    a.run(fused=False)
    b.run(fused=True)
    ya, yb = a.y_view.float(), b.y_view.float()
    assert torch.all((ya - yb).abs() <= 1e-2 + 1e-2 * ya.abs())
    rows = lora_rows(wl.mapping, wl.shape.num_tokens, wl.shape.max_loras)
    ua, ub = a.u.view[:, rows], b.u.view[:, rows]
    assert torch.all((ua - ub).abs() <= 1e-2 + 1e-2 * ua.abs())


def test_shrink_expand_one_call_in_a_graph_with_new_mappings(dev):
    sh = W.custom_shape(max_num_tokens=256, num_tokens=256, hidden=2048,
                        slice_widths=(1024, 1024, 1024), max_loras=8, rank=8, neg_prob=0.1)
    rng = np.random.default_rng(21)
    layer = W.make_layer(sh, rng)
    g_case = DeviceCase(sh, W.make_mapping(sh, rng), layer, dev)
    stream = torch.cuda.Stream()
    y_clean = g_case.y.view.clone()
    with torch.cuda.stream(stream):
        g_case.prepare(stream); g_case.shrink_expand(stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        g_case.prepare(stream)
        g_case.shrink_expand(stream)
    for trial, n_new in enumerate((256, 100, 17)):
        sh2 = W.custom_shape(max_num_tokens=256, num_tokens=n_new, hidden=2048,
                             slice_widths=(1024, 1024, 1024), max_loras=8, rank=8, neg_prob=0.2)
        m_new = W.make_mapping(sh2, np.random.default_rng(300 + trial))
        g_case.mapping.copy_(torch.from_numpy(m_new))
        g_case.n.fill_(n_new)
        g_case.y.view.copy_(y_clean)
        g_case.u.view.view(torch.int32).fill_(U_SENTINEL_BITS)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        eager = DeviceCase(sh2, m_new, layer, dev)
        eager.run(fused=True)
        assert torch.equal(g_case.y.view.view(torch.int16), eager.y.view.view(torch.int16))
        assert torch.equal(g_case.u.view.view(torch.int32), eager.u.view.view(torch.int32))


# ------------------------------------------------------------ one-call split-K path

# hidden sizes above 8192 keep these shapes off the single-wave fused kernel
# (more than 16 k-blocks per CTA), so the one call takes the split-K path
SPLIT_SHAPES = [
    ("decode_qkv", None),
    ("ragged3", (300, 211, 8208, (264, 72, 136), 6, 8)),
    ("rank16", (256, 256, 9216, (512, 512), 4, 16)),
    ("rank32", (1000, 977, 8264, (1032, 520, 264), 5, 32)),
    ("many_loras", (512, 500, 8200, (1024,), 64, 8)),
]


def _split_case(name, spec, dev):
    if spec is None:
        wl = W.make_workload(name)
        return DeviceCase(wl.shape, wl.mapping, wl.layers[0], dev, split_workspace=True)
    T, n, H, widths, L, R = spec
    shape = W.custom_shape(max_num_tokens=T, num_tokens=n, hidden=H, slice_widths=widths,
                           max_loras=L, rank=R, neg_prob=0.15)
    rng = np.random.default_rng(T + R + 7)
    return DeviceCase(shape, W.make_mapping(shape, rng), W.make_layer(shape, rng), dev,
                      split_workspace=True)


def _path_of(case):
    sh = case.shape
    return binding.lora_shrink_expand_path(sh.max_num_tokens, sh.max_loras, sh.hidden,
                                           sh.slice_widths, sh.rank, case.ws.view.numel(),
                                           fp16=case.f16, paged=case.paged)


@pytest.mark.parametrize("name,spec", SPLIT_SHAPES)
def test_split_k_one_call_matches_the_oracle(name, spec, dev):
    case = _split_case(name, spec, dev)
    assert case.ws.view.numel() > case.ws_base  # the larger workspace was offered
    assert _path_of(case) == binding.LORA_PATH_SPLIT_PAIR
    check_case(case, fused=True)   # every adapter row
    # the split-K path ran: its partial tiles landed behind the metadata
    assert torch.any(case.ws.view[case.ws_base:] != 0)


def _close_to_the_two_calls(a, b):
    """The split-K one call against lora_shrink + lora_expand: the same fp32
    products summed in another grouping, so u agrees to fp32 rounding and y
    to one bf16 rounding step; untouched rows stay bit-identical."""
    ua, ub = a.u.view.double(), b.u.view.double()
    rows = lora_rows(a.mapping_np, a.shape.num_tokens, a.shape.max_loras)
    assert torch.all((ua[:, rows] - ub[:, rows]).abs() <= 1e-6 + 1e-5 * ua[:, rows].abs())
    keep = np.ones(a.shape.max_num_tokens, bool)
    keep[rows] = False
    assert torch.equal(a.u.view.view(torch.int32)[:, keep], b.u.view.view(torch.int32)[:, keep])
    ya, yb = a.y.view[rows].double(), b.y.view[rows].double()
    assert torch.all((ya - yb).abs() <= 1e-3 + 2.0 ** -7 * ya.abs())
    assert torch.equal(a.y.view.view(torch.int16)[keep], b.y.view.view(torch.int16)[keep])


@pytest.mark.parametrize("name,spec", SPLIT_SHAPES[:3])
def test_split_k_one_call_agrees_with_the_two_calls(name, spec, dev):
    a = _split_case(name, spec, dev)
    b = _split_case(name, spec, dev)
    a.run(fused=False)
    b.run(fused=True)
    assert torch.any(b.ws.view[b.ws_base:] != 0)
    _close_to_the_two_calls(a, b)


def test_split_k_one_call_in_a_graph_with_new_mappings(dev):
    sh = W.custom_shape(max_num_tokens=256, num_tokens=256, hidden=8200,
                        slice_widths=(1024, 1024, 1024), max_loras=8, rank=8, neg_prob=0.1)
    rng = np.random.default_rng(23)
    layer = W.make_layer(sh, rng)
    g_case = DeviceCase(sh, W.make_mapping(sh, rng), layer, dev, split_workspace=True)
    stream = torch.cuda.Stream()
    y_clean = g_case.y.view.clone()
    with torch.cuda.stream(stream):
        g_case.prepare(stream); g_case.shrink_expand(stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        g_case.prepare(stream)
        g_case.shrink_expand(stream)
    for trial, n_new in enumerate((256, 100, 17, 0)):
        sh2 = W.custom_shape(max_num_tokens=256, num_tokens=n_new, hidden=8200,
                             slice_widths=(1024, 1024, 1024), max_loras=8, rank=8, neg_prob=0.2)
        m_new = W.make_mapping(sh2, np.random.default_rng(400 + trial))
        g_case.mapping.copy_(torch.from_numpy(m_new))
        g_case.n.fill_(n_new)
        g_case.y.view.copy_(y_clean)
        g_case.u.view.view(torch.int32).fill_(U_SENTINEL_BITS)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        eager = DeviceCase(sh2, m_new, layer, dev, split_workspace=True)
        eager.run(fused=True)
        assert torch.equal(g_case.y.view.view(torch.int16), eager.y.view.view(torch.int16))
        assert torch.equal(g_case.u.view.view(torch.int32), eager.u.view.view(torch.int32))


@pytest.mark.parametrize("name,spec", SPLIT_SHAPES[:2])
def test_split_k_halves_equal_the_one_call(name, spec, dev):
    a = _split_case(name, spec, dev)
    b = _split_case(name, spec, dev)
    a.run(fused=True)
    b.prepare()
    binding.lora_shrink_partials(b.x, b.a, b.sorted.view, b.starts.view, b.ws.view)
    binding.lora_expand_partials(b.shape.hidden, b.b, b.shape.scale, b.u.view, b.y_view,
                                 b.sorted.view, b.starts.view, b.ws.view)
    torch.cuda.synchronize()
    assert b.guards_intact()
    assert torch.equal(a.y.view.view(torch.int16), b.y.view.view(torch.int16))
    assert torch.equal(a.u.view.view(torch.int32), b.u.view.view(torch.int32))


# ------------------------------------------------------------ per-adapter scales

def _scaled_case(spec, dev, split_workspace=False, seed=31):
    T, n, H, widths, L, R = spec
    shape = W.custom_shape(max_num_tokens=T, num_tokens=n, hidden=H, slice_widths=widths,
                           max_loras=L, rank=R, scale=0.5, neg_prob=0.15)
    rng = np.random.default_rng(seed)
    factors = rng.uniform(-2.0, 2.0, L).astype(np.float32)
    factors[0] = 0.0  # one adapter switched off
    return DeviceCase(shape, W.make_mapping(shape, rng), W.make_layer(shape, rng), dev,
                      split_workspace=split_workspace, lora_scales=factors)


SCALED_SHAPES = [
    ("two_calls_cluster", (300, 280, 1032, (520, 264), 6, 16), False, False),
    ("one_call_fused", (64, 64, 512, (512,), 4, 8), False, True),
    ("one_call_split_k", (256, 240, 8200, (1024, 1024, 1024), 4, 8), True, True),
    ("one_call_cluster_large", (2048, 2000, 1024, (2048,), 8, 64), False, True),
]


@pytest.mark.parametrize("name,spec,split_ws,one_call", SCALED_SHAPES)
def test_per_adapter_scales_match_the_oracle(name, spec, split_ws, one_call, dev):
    case = _scaled_case(spec, dev, split_workspace=split_ws)
    check_case(case, fused=one_call)
    if split_ws:
        assert torch.any(case.ws.view[case.ws_base:] != 0)


def test_per_adapter_scales_of_one_equal_no_scales(dev):
    spec = (256, 240, 1024, (512, 512, 512), 4, 8)
    a = _scaled_case(spec, dev)
    b = _scaled_case(spec, dev)
    a.lora_scales.fill_(1.0)
    b.lora_scales = None
    a.run()
    b.run()
    assert torch.equal(a.u.view.view(torch.int32), b.u.view.view(torch.int32))
    assert torch.equal(a.y.view.view(torch.int16), b.y.view.view(torch.int16))


# ------------------------------------------------------------ paged adapter weights

PAGED_SHAPES = [
    # (spec, split_workspace, one_call)
    ("decode_like_two_calls", (256, 240, 1032, (512, 264, 136), 4, 8), False, False),
    ("decode_like_split_k", (256, 240, 8200, (1024, 1024, 1024), 4, 8), True, True),
    ("prefill_like_cluster", (2048, 2000, 1024, (1024,), 8, 16), False, True),
    ("rank128", (512, 500, 512, (256,), 6, 128), False, False),
    ("tiny_one_call", (64, 64, 512, (512,), 4, 8), False, True),
    ("prefill_k_groups", (2048, 2000, 2120, (264,), 6, 16), False, False),
    ("prefill_k_groups_one_call", (2048, 2000, 2120, (264,), 6, 16), False, True),
]


def _paged_case(spec, dev, split_workspace=False, seed=41, paged=True):
    T, n, H, widths, L, R = spec
    shape = W.custom_shape(max_num_tokens=T, num_tokens=n, hidden=H, slice_widths=widths,
                           max_loras=L, rank=R, neg_prob=0.15)
    rng = np.random.default_rng(seed)
    return DeviceCase(shape, W.make_mapping(shape, rng), W.make_layer(shape, rng), dev,
                      split_workspace=split_workspace, paged=paged)


@pytest.mark.parametrize("name,spec,split_ws,one_call", PAGED_SHAPES)
def test_paged_weights_match_the_oracle(name, spec, split_ws, one_call, dev):
    case = _paged_case(spec, dev, split_workspace=split_ws)
    check_case(case, fused=one_call)
    assert case.ws.view[:4].view(torch.int32).item() & binding.LORA_STATUS_BAD_WEIGHT == 0


@pytest.mark.parametrize("name,spec,split_ws,one_call", PAGED_SHAPES[:3])
def test_paged_weights_equal_stacked_weights_bit_for_bit(name, spec, split_ws, one_call, dev):
    a = _paged_case(spec, dev, split_workspace=split_ws, paged=True)
    b = _paged_case(spec, dev, split_workspace=split_ws, paged=False)
    a.run(fused=one_call)
    b.run(fused=one_call)
    assert torch.equal(a.u.view.view(torch.int32), b.u.view.view(torch.int32))
    assert torch.equal(a.y.view.view(torch.int16), b.y.view.view(torch.int16))


def test_paged_zero_and_misaligned_entries_read_as_zero_adapters(dev):
    spec = (256, 256, 1024, (512, 512), 4, 16)
    case = _paged_case(spec, dev)
    # adapter 1: no pages (0); adapter 2: misaligned addresses
    for tab in case.a_tables + case.b_tables:
        tab[1] = 0
        tab[2] = tab[2] + 2
    lay = case.layer
    for s in range(case.shape.num_slices):
        lay.lora_a[s][1:3] = 0
        lay.lora_b[s][1:3] = 0
    check_case(case)
    assert case.ws.view[:4].view(torch.int32).item() & binding.LORA_STATUS_BAD_WEIGHT


# ------------------------------------------------------------ fp16 inputs

F16_SHAPES = [
    # (name, spec or workload, split_workspace, one_call)
    ("decode_qkv_two_calls", None, False, False),
    ("decode_qkv_split_k", None, True, True),
    ("tiny_fused", (64, 64, 512, (512,), 4, 8), False, True),
    ("ragged_cluster", (300, 211, 1032, (264, 72, 136), 6, 16), False, True),
    ("prefill_like", (4096, 4000, 1024, (1024,), 8, 16), False, False),
    ("rank64_two_slices", (1024, 1000, 1024, (1032, 520), 8, 64), False, True),
    ("rank128", (512, 500, 2048, (256,), 6, 128), False, False),
    ("split_k_rank32", (1000, 977, 8264, (1032, 520, 264), 5, 32), True, True),
    ("prefill_k_groups", (2048, 1990, 2120, (264, 136), 6, 8), False, False),
    ("prefill_k_groups_one_call", (2048, 1990, 2120, (264, 136), 6, 8), False, True),
]


def _f16_case(spec, dev, split_workspace=False, seed=51, lora_scales=None):
    if spec is None:
        wl = W.make_workload("decode_qkv")
        return DeviceCase(wl.shape, wl.mapping, wl.layers[0], dev,
                          split_workspace=split_workspace, f16=True, lora_scales=lora_scales)
    T, n, H, widths, L, R = spec
    shape = W.custom_shape(max_num_tokens=T, num_tokens=n, hidden=H, slice_widths=widths,
                           max_loras=L, rank=R, scale=0.5, neg_prob=0.15)
    rng = np.random.default_rng(seed)
    return DeviceCase(shape, W.make_mapping(shape, rng), W.make_layer(shape, rng), dev,
                      split_workspace=split_workspace, f16=True, lora_scales=lora_scales)


@pytest.mark.parametrize("name,spec,split_ws,one_call", F16_SHAPES)
def test_fp16_inputs_match_the_oracle(name, spec, split_ws, one_call, dev):
    case = _f16_case(spec, dev, split_workspace=split_ws)
    assert case.x.dtype == torch.float16 and case.y_view.dtype == torch.float16
    check_case(case, fused=one_call)
    if split_ws:
        assert torch.any(case.ws.view[case.ws_base:] != 0)


def test_fp16_inputs_with_per_adapter_scales(dev):
    spec = (256, 240, 8200, (1024, 512), 4, 8)
    factors = np.array([0.0, 1.5, -0.75, 2.0], np.float32)
    case = _f16_case(spec, dev, split_workspace=True, lora_scales=factors)
    check_case(case, fused=True)


@pytest.mark.parametrize("one_call", [False, True])
def test_fp16_and_bf16_paths_agree_exactly_on_small_integers(one_call, dev):
    """Small integers are exact in both formats and every product and sum
    stays exact in fp32, so the two input types give the same values."""
    T, H = 64, 4096
    case_b, _ = _int_case(dev, T, H, 16, seed=H)
    case_h = DeviceCase(case_b.shape, case_b.mapping_np, case_b.layer, dev, f16=True)
    case_b.run(fused=one_call)
    case_h.run(fused=one_call)
    assert torch.equal(case_b.u.view.view(torch.int32), case_h.u.view.view(torch.int32))
    rows = lora_rows(case_b.mapping_np, T, 3)
    assert torch.equal(case_b.y.view[rows].float(), case_h.y.view[rows].float())


def test_fp16_split_k_halves_equal_the_one_call(dev):
    a = _f16_case(None, dev, split_workspace=True)
    b = _f16_case(None, dev, split_workspace=True)
    a.run(fused=True)
    b.prepare()
    binding.lora_shrink_partials(b.x, b.a, b.sorted.view, b.starts.view, b.ws.view)
    binding.lora_expand_partials(b.shape.hidden, b.b, b.shape.scale, b.u.view, b.y_view,
                                 b.sorted.view, b.starts.view, b.ws.view)
    torch.cuda.synchronize()
    assert b.guards_intact()
    assert torch.equal(a.y.view.view(torch.int16), b.y.view.view(torch.int16))
    assert torch.equal(a.u.view.view(torch.int32), b.u.view.view(torch.int32))


# ------------------------------------------------------------ the LoRA delta, tightly

def _zero_base_case(dev, workload=None, spec=None, **kw):
    """A case whose base output y is zero, so y after the call is the LoRA delta."""
    if workload is not None:
        wl = W.make_workload(workload)
        shape, mapping, layer = wl.shape, wl.mapping, wl.layers[0]
    else:
        T, n, H, widths, L, R = spec
        shape = W.custom_shape(max_num_tokens=T, num_tokens=n, hidden=H, slice_widths=widths,
                               max_loras=L, rank=R, neg_prob=0.15)
        rng = np.random.default_rng(T + H + R)
        mapping, layer = W.make_mapping(shape, rng), W.make_layer(shape, rng)
    layer = W.Layer(x=layer.x, lora_a=layer.lora_a, lora_b=layer.lora_b,
                    y=np.zeros_like(layer.y))
    return DeviceCase(shape, mapping, layer, dev, **kw)


ZERO_BASE_PATHS = [
    # (name, workload, spec, one_call, DeviceCase options)
    ("two_calls_decode", "decode_qkv", None, False, {}),
    ("fused_tiny", "tiny", None, True, {}),
    ("split_k_decode", "decode_qkv", None, True, {"split_workspace": True}),
    ("cluster_one_call_prefill", "chunked_prefill", None, True, {}),
    ("cluster_one_call_gate_up", "mlp_gate_up", None, True, {}),
    ("cluster_one_call_down_proj", "down_proj_graph", None, True, {}),
    ("paged_one_call", None, (256, 240, 1032, (512, 264, 136), 4, 8), True, {"paged": True}),
    ("paged_rank128", None, (512, 500, 512, (256,), 6, 128), False, {"paged": True}),
    ("fp16_split_k", "decode_qkv", None, True, {"split_workspace": True, "f16": True}),
    ("fp16_rank64", None, (1024, 1000, 1024, (1032, 520), 8, 64), True, {"f16": True}),
]


@pytest.mark.parametrize("name,workload,spec,one_call,opts", ZERO_BASE_PATHS)
def test_zero_base_output_holds_the_delta_tightly(name, workload, spec, one_call, opts, dev):
    """With a zero base output, y after the call is the LoRA delta, whose
    values (std about 0.07) sit far below the 1e-2 absolute term of the
    general bar.  The delta's own error is one final rounding (2^-9 relative
    for bf16, 2^-12 for fp16) plus the fp32 sums and the 16-bit split of u
    (about 2^-17 relative per term), so it is held to 2^-7 |delta| + 1e-4
    (bf16) or 2^-9 |delta| + 1e-4 (fp16) on every element."""
    case = _zero_base_case(dev, workload, spec, **opts)
    sh, lay = case.shape, case.layer
    case.run(fused=one_call)
    if opts.get("split_workspace"):
        assert torch.any(case.ws.view[case.ws_base:] != 0)   # the split-K path ran
    rows = lora_rows(case.mapping_np, sh.num_tokens, sh.max_loras)
    f16 = case.f16
    u_ref = oracle.shrink(lay.x, lay.lora_a, sh.scale, case.mapping_np, sh.num_tokens,
                          sh.max_loras, u_init=np.zeros((sh.num_slices, sh.max_num_tokens,
                                                         sh.rank)), f16=f16)
    d_ref = oracle.expand(u_ref, lay.lora_b, np.ascontiguousarray(lay.y), case.mapping_np,
                          sh.num_tokens, sh.max_loras, f16=f16)[rows]
    d = oracle.decode_bits(bits_of(case.y_view), f16=f16)[rows]
    bound = (2.0 ** -9 if f16 else 2.0 ** -7) * np.abs(d_ref) + 1e-4
    err = np.abs(d - d_ref)
    assert np.all(err <= bound), f"worst err/bound {float(np.max(err / bound)):.3f}"
    assert np.all(case.y_view.float().cpu().numpy()[np.setdiff1d(
        np.arange(sh.max_num_tokens), rows)] == 0)


# ------------------------------------------------------------ stream ordering

@pytest.mark.parametrize("one_call", [False, True])
def test_weights_rewritten_right_before_the_call_are_used(one_call, dev):
    """A torch copy kernel rewrites adapter 1's A and B on the stream right
    before the call: the kernels copy nothing into shared memory before their
    dependency wait (only L2 prefetches), so they compute with the new weights."""
    shape = W.custom_shape(max_num_tokens=256, num_tokens=256, hidden=1024,
                           slice_widths=(512, 256), max_loras=4, rank=16, neg_prob=0.1)
    case = make_case(shape, dev, seed=61)
    rng = np.random.default_rng(62)
    new_a = [W.f32_to_bf16_bits(rng.standard_normal((16, 1024), dtype=np.float32) * 0.02)
             for _ in range(2)]
    new_b = [W.f32_to_bf16_bits(rng.standard_normal((16, w), dtype=np.float32) * 0.02)
             for w in (512, 256)]
    staged_a = [bf16_dev(v, dev) for v in new_a]
    staged_b = [bf16_dev(v, dev) for v in new_b]
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        case.prepare(stream)
        for s_ in range(2):
            case.a[s_][1].copy_(staged_a[s_])
            case.b[s_][1].copy_(staged_b[s_])
        if one_call:
            case.shrink_expand(stream)
        else:
            case.shrink(stream)
            case.expand(stream)
    torch.cuda.synchronize()
    lay = case.layer
    for s_ in range(2):
        lay.lora_a[s_][1] = new_a[s_]
        lay.lora_b[s_][1] = new_b[s_]
    sh = case.shape
    rows = lora_rows(case.mapping_np, sh.num_tokens, sh.max_loras)
    assert np.any(case.mapping_np[rows] == 1)
    u_ref = oracle.shrink(lay.x, lay.lora_a, sh.scale, case.mapping_np, sh.num_tokens,
                          sh.max_loras, u_init=np.zeros((2, 256, 16)))
    y_ref = oracle.expand(u_ref, lay.lora_b, case.y_in_bits, case.mapping_np, sh.num_tokens,
                          sh.max_loras)
    ok_u, r_u = within_tol(case.u.view.cpu().numpy()[:, rows].astype(np.float64), u_ref[:, rows])
    assert ok_u, r_u
    y = oracle.bf16_bits_to_f64(bits_of(case.y.view))
    ok_y, r_y = within_tol(y[rows], y_ref[rows])
    assert ok_y, r_y


@pytest.mark.parametrize("one_call", [False, True])
def test_batch_without_adapter_tokens_after_a_kernel_that_writes_y(one_call, dev):
    """No token has an adapter, so no CTA of the shrink or expand has work;
    the y a preceding kernel wrote must come out unchanged."""
    shape = W.custom_shape(max_num_tokens=256, num_tokens=256, hidden=4096,
                           slice_widths=(4096, 4096, 4096), max_loras=4, rank=8, neg_prob=1.0)
    case = make_case(shape, dev, seed=63, split_workspace=one_call)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        case.y_view.fill_(1.5)
        case.prepare(stream)
        if one_call:
            case.shrink_expand(stream)
        else:
            case.shrink(stream)
            case.expand(stream)
        after = case.y_view.clone()
    torch.cuda.synchronize()
    assert torch.all(after == 1.5)
    assert torch.all(case.u.view.view(torch.int32) == U_SENTINEL_BITS)


# ------------------------------------------------------------ one-call paths

def test_path_query_names_each_path(dev):
    """lora_shrink_expand_path: decode takes the split-K pair with the larger
    workspace and the cluster pair without it; tiny batches the fused kernel
    (never with paged weights); prefill the cluster pair."""
    q = binding.lora_shrink_expand_path
    dq = W.CONFIGS["decode_qkv"]
    big = binding.lora_shrink_expand_workspace_size(256, 4, 4096, dq.slice_widths, 8)
    base = binding.lora_workspace_size(256, 4)
    assert q(256, 4, 4096, dq.slice_widths, 8, big) == binding.LORA_PATH_SPLIT_PAIR
    assert q(256, 4, 4096, dq.slice_widths, 8, big, fp16=True) == binding.LORA_PATH_SPLIT_PAIR
    assert q(256, 4, 4096, dq.slice_widths, 8, base) == binding.LORA_PATH_PAIR
    assert q(256, 4, 4096, dq.slice_widths, 8, big, paged=True) == binding.LORA_PATH_SPLIT_PAIR
    tiny_ws = binding.lora_workspace_size(64, 4)
    assert q(64, 4, 512, (512,), 8, tiny_ws) == binding.LORA_PATH_FUSED
    assert q(64, 4, 512, (512,), 8, tiny_ws, paged=True) == binding.LORA_PATH_PAIR
    pf = W.CONFIGS["chunked_prefill"]
    assert q(8192, 8, 4096, pf.slice_widths, 16,
             binding.lora_workspace_size(8192, 8)) == binding.LORA_PATH_PAIR


def _layer_case(T, n, H, widths, L, R, seed, dev, ws_bytes):
    shape = W.custom_shape(max_num_tokens=T, num_tokens=n, hidden=H, slice_widths=widths,
                           max_loras=L, rank=R, neg_prob=0.1)
    rng = np.random.default_rng(seed)
    case = DeviceCase(shape, W.make_mapping(shape, rng), W.make_layer(shape, rng), dev)
    case.ws = type(case.ws)((ws_bytes,), torch.uint8, dev, fill_bits=0)
    return case


def test_split_k_layers_of_different_splits_share_a_workspace(dev):
    """Layers of different hidden sizes (splits of 16 and 8) run one after
    the other on one workspace, as a model's LoRA layers share one grouping:
    each call's partial tiles overwrite the previous call's, and every call
    gives the results of the two split-K halves run on a workspace of its
    own bit for bit."""
    # 16 adapters and wide slices keep the batch off the fused kernel; hidden
    # 3072 gives 48 k-blocks (a split of 8), hidden 4096 64 (a split of 16)
    T, n, L, R, widths = 256, 250, 16, 8, (8192, 4096, 4096)
    hs = (4096, 3072, 4096)
    ws_bytes = max(binding.lora_shrink_expand_workspace_size(T, L, H, widths, R) for H in hs)
    layers = [_layer_case(T, n, H, widths, L, R, 70 + i, dev, ws_bytes)
              for i, H in enumerate(hs)]
    for c in layers:
        assert _path_of(c) == binding.LORA_PATH_SPLIT_PAIR, c.shape.hidden
    m = layers[0]
    for c in layers[1:]:   # one batch: the same mapping for every layer
        c.mapping.copy_(m.mapping)
        c.mapping_np = m.mapping_np
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        binding.lora_prepare_metadata(m.mapping, m.n, L, m.sorted.view, m.counts.view,
                                      m.starts.view, m.ws.view, stream)
        for c in layers:
            binding.lora_shrink_expand(c.x, c.a, c.b, c.shape.scale, c.u.view, c.y_view,
                                       m.sorted.view, m.starts.view, m.ws.view, stream)
    torch.cuda.synchronize()
    for i, c in enumerate(layers):
        ref = _layer_case(T, n, c.shape.hidden, widths, L, R, 70 + i, dev, ws_bytes)
        ref.mapping.copy_(m.mapping)
        ref.prepare()
        binding.lora_shrink_partials(ref.x, ref.a, ref.sorted.view, ref.starts.view, ref.ws.view)
        binding.lora_expand_partials(ref.shape.hidden, ref.b, ref.shape.scale, ref.u.view,
                                     ref.y_view, ref.sorted.view, ref.starts.view, ref.ws.view)
        torch.cuda.synchronize()
        assert torch.equal(c.y.view.view(torch.int16), ref.y.view.view(torch.int16)), i
        assert torch.equal(c.u.view.view(torch.int32), ref.u.view.view(torch.int32)), i
    assert m.ws.view[:4].view(torch.int32).item() == 0   # status clean


# ------------------------------------------------------------ the tcgen05 expand (ranks 64 / 128)

# more than 1024 tokens and rank 128: lora_expand runs the tcgen05 kernel
# (128-token tiles, 128-column blocks, accumulators in tensor memory); the
# rank-64 shapes run the mma.sync kernel beside them
TC_SHAPES = [
    # (T, n, H, widths, L, R)
    (2048, 1900, 512, (1032, 520, 264), 5, 128),  # three slices, partial column blocks
    (1100, 1100, 256, (128,), 3, 128),            # one column block, ragged tiles
    (4096, 3000, 384, (2048,), 40, 128),          # many adapters, mostly partial tiles
    (1536, 1536, 1024, (264, 136), 2, 128),       # few adapters, several full tiles each
    (2048, 1900, 512, (1032, 520, 264), 5, 64),   # rank 64: the mma.sync kernel
]


@pytest.mark.parametrize("one_call", [False, True])
@pytest.mark.parametrize("T,n,H,widths,L,R", TC_SHAPES)
def test_tcgen05_expand_matches_the_oracle(T, n, H, widths, L, R, one_call, dev):
    shape = W.custom_shape(max_num_tokens=T, num_tokens=n, hidden=H, slice_widths=widths,
                           max_loras=L, rank=R, neg_prob=0.15)
    check_case(make_case(shape, dev, seed=T + R + len(widths)), fused=one_call)


@pytest.mark.parametrize("T,n,H,widths,L,R", TC_SHAPES[:2])
def test_tcgen05_expand_fp16_inputs(T, n, H, widths, L, R, dev):
    shape = W.custom_shape(max_num_tokens=T, num_tokens=n, hidden=H, slice_widths=widths,
                           max_loras=L, rank=R, scale=0.5, neg_prob=0.15)
    rng = np.random.default_rng(T + 5)
    case = DeviceCase(shape, W.make_mapping(shape, rng), W.make_layer(shape, rng), dev, f16=True)
    check_case(case, fused=True)


@pytest.mark.parametrize("R", [128])
def test_tcgen05_expand_small_integers_are_bit_exact(R, dev):
    """Integer x, A, B and y keep u and every partial sum of the expand exact
    in fp32 whatever the summation order, so the tensor-memory accumulation
    must give the oracle's exact y rounded once to bf16 (round to nearest
    even; sums of up to 128 terms can exceed bf16's exact integers), bit for
    bit, and the oracle's u exactly."""
    T, H = 1100, 64
    case, (xi, ai, bi, yi, m) = _int_case(dev, T, H, 16, seed=R, R=R, widths=(136, 264))
    case.run()
    u_ref = oracle.shrink(case.layer.x, case.layer.lora_a, 0.5, m, T, 3,
                          u_init=np.zeros((2, T, R)))
    y_ref = oracle.expand(u_ref, case.layer.lora_b, case.layer.y, m, T, 3)
    assert np.all(np.abs(y_ref) < 2 ** 24) and np.array_equal(y_ref, np.round(y_ref))
    rows = lora_rows(m, T, 3)
    assert np.array_equal(case.u.view.cpu().numpy()[:, rows].astype(np.float64), u_ref[:, rows])
    assert np.array_equal(bits_of(case.y.view), W.f32_to_bf16_bits(y_ref.astype(np.float32)))


def test_tcgen05_expand_alone_equals_the_oracle_on_the_gpu_u(dev):
    """The expand by itself on a u the test writes (every row of every slice
    set, not only adapter rows): only adapter rows of y change, by exactly the
    oracle's expand of that u within the bar."""
    shape = W.custom_shape(max_num_tokens=2048, num_tokens=2000, hidden=64,
                           slice_widths=(1024, 512), max_loras=6, rank=128, neg_prob=0.2)
    case = make_case(shape, dev, seed=91)
    case.prepare()
    rng = np.random.default_rng(92)
    u = rng.standard_normal((2, 2048, 128)).astype(np.float32)
    case.u.view.copy_(torch.from_numpy(u))
    case.expand()
    torch.cuda.synchronize()
    y_ref = oracle.expand(u.astype(np.float64), case.layer.lora_b, case.y_in_bits[:, :1536],
                          case.mapping_np, 2000, 6)
    y = oracle.bf16_bits_to_f64(bits_of(case.y_view))
    rows = lora_rows(case.mapping_np, 2000, 6)
    ok, worst = within_tol(y[rows], y_ref[rows])
    assert ok, worst
    keep = np.setdiff1d(np.arange(2048), rows)
    assert np.array_equal(bits_of(case.y.view)[keep], case.y_in_bits[keep])
    assert case.guards_intact()
