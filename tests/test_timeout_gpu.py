"""The kernels' bounded waits, made to run out on purpose through the test
hook of include/gathered_rank_gemm_testing.h (one barrier arrival too many,
no copy issued, a 1 ms limit).  On every path (the two calls, the fused
kernel, the split-K pair, the tcgen05 expand, the shrink's stages of four
k-blocks) the call must finish, report
LORA_STATUS_TIMEOUT, write no output, leave every guard band alone, and leave
the GPU and the buffers fit for the next call, which must match the oracle."""
import numpy as np
import pytest

from gathered_rank_gemm_gb300 import binding
from gathered_rank_gemm_gb300 import workloads as W

from helpers import DeviceCase, U_SENTINEL_BITS, bits_of, check_case

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


class timeouts_injected:
    def __enter__(self):
        assert binding.lora_testing_inject_timeout(True) is False
        return self

    def __exit__(self, *exc):
        assert binding.lora_testing_inject_timeout(False) is True
        return False


def _custom(dev, T, n, H, widths, L, R, split_workspace=False):
    shape = W.custom_shape(max_num_tokens=T, num_tokens=n, hidden=H, slice_widths=widths,
                           max_loras=L, rank=R, neg_prob=0.1)
    rng = np.random.default_rng(T + R + len(widths))
    return DeviceCase(shape, W.make_mapping(shape, rng), W.make_layer(shape, rng), dev,
                      split_workspace=split_workspace)


def _named(dev, name, split_workspace=False):
    wl = W.make_workload(name)
    return DeviceCase(wl.shape, wl.mapping, wl.layers[0], dev, split_workspace=split_workspace)


def _path(case):
    sh = case.shape
    return binding.lora_shrink_expand_path(sh.max_num_tokens, sh.max_loras, sh.hidden,
                                           sh.slice_widths, sh.rank, case.ws.view.numel())


CASES = [
    # (name, builder, one call, expected one-call path)
    ("two calls, 16-token tiles", lambda d: _custom(d, 256, 250, 2048, (512,), 4, 16), False, None),
    ("two calls, 64-token tiles", lambda d: _custom(d, 1100, 1100, 4096, (1024, 512), 6, 64),
     False, None),
    ("fused kernel", lambda d: _named(d, "tiny"), True, binding.LORA_PATH_FUSED),
    ("split-K pair", lambda d: _named(d, "decode_qkv", split_workspace=True), True,
     binding.LORA_PATH_SPLIT_PAIR),
    ("cluster pair", lambda d: _custom(d, 1100, 1100, 1032, (520, 264), 3, 16), True,
     binding.LORA_PATH_PAIR),
    ("tcgen05 expand", lambda d: _custom(d, 2048, 1900, 512, (1032, 520, 264), 5, 128), False,
     None),
    # 32-token tiles of rank 16 over 34 k-blocks: stages of four k-blocks, the
    # last short (lora_shrink, and the shrink of the cluster pair)
    ("two calls, four-k-block stages", lambda d: _custom(d, 1100, 1100, 2120, (264,), 4, 16),
     False, None),
    ("cluster pair, four-k-block stages",
     lambda d: _custom(d, 1100, 1100, 2120, (264,), 4, 16), True, binding.LORA_PATH_PAIR),
]


@pytest.mark.parametrize("name,build_case,one_call,path", CASES, ids=[c[0] for c in CASES])
def test_timeout_is_reported_writes_nothing_and_the_next_call_is_whole(
        name, build_case, one_call, path, dev):
    case = build_case(dev)
    if path is not None:
        assert _path(case) == path
    case.prepare()
    torch.cuda.synchronize()
    assert binding.lora_read_status(case.ws.view) == 0
    with timeouts_injected():
        if one_call:
            case.shrink_expand()
        else:
            case.shrink()
            case.expand()
        torch.cuda.synchronize()
    assert binding.lora_read_status(case.ws.view) & binding.LORA_STATUS_TIMEOUT
    u_bits = case.u.view.cpu().numpy().view(np.uint32)
    assert np.all(u_bits == U_SENTINEL_BITS), "a timed-out call wrote u"
    assert np.array_equal(bits_of(case.y.view), case.y_in_bits), "a timed-out call wrote y"
    assert case.guards_intact()
    # the next call, with the hook off, on the same buffers, matches the oracle
    check_case(case, fused=one_call)
    assert binding.lora_read_status(case.ws.view) == 0
