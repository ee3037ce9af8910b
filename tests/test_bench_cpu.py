"""CPU checks of bench.py's bookkeeping: the algorithmic bytes of the roofline
and the committed DRAM-traffic records it reports (no GPU needed)."""
import json
import os

import numpy as np

import bench
from gathered_rank_gemm_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _count_bytes(shape, mapping):
    """Per-token / per-adapter byte count written as loops (a second route to
    the same quantity): every adapter token reads its x row and writes its u
    rows (shrink), reads its u rows and reads + writes its y row (expand);
    every adapter with a token is read once per step."""
    n, L = shape.num_tokens, shape.max_loras
    S, R, H, N = shape.num_slices, shape.rank, shape.hidden, shape.out_width
    shrink = expand = 0
    active = set()
    for t in range(n):
        lid = int(mapping[t])
        if not 0 <= lid < L:
            continue
        active.add(lid)
        shrink += 2 * H + S * R * 4
        expand += S * R * 4 + 2 * (2 * N)
    for _ in active:
        shrink += sum(R * H * 2 for _ in range(S))
        expand += sum(R * w * 2 for w in shape.slice_widths)
    return shrink, expand


def test_algorithmic_bytes_match_a_token_by_token_count():
    for name in ("tiny", "decode_qkv", "chunked_prefill", "down_proj_graph"):
        wl = W.make_workload(name, num_layers=0)
        alg = bench.algorithmic_bytes(wl.shape, wl.mapping)
        assert (alg["shrink"], alg["expand"]) == _count_bytes(wl.shape, wl.mapping)


def test_decode_and_prefill_bytes_per_launch():
    """The per-launch figures the roofline divides by (one layer of one batch)."""
    d = W.make_workload("decode_qkv", num_layers=0)
    a = bench.algorithmic_bytes(d.shape, d.mapping)
    assert (a["n_lora_tokens"], a["active_loras"]) == (235, 4)
    assert (a["shrink"], a["expand"]) == (2_734_112, 12_359_712)
    p = W.make_workload("chunked_prefill", num_layers=0)
    b = bench.algorithmic_bytes(p.shape, p.mapping)
    assert (b["shrink"], b["expand"]) == (68_681_728, 135_790_592)


def test_recorded_traffic_is_returned_only_for_unchanged_kernels():
    """The DRAM traffic the bench reports comes from committed ncu records:
    a record whose source hash matches the kernel sources is returned, a
    stale one reads as null."""
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        rec = json.load(f)
    assert rec
    for key, r in rec.items():
        kernel, workload = key.split("/")
        assert r["bytes_per_launch"] == r["read"] + r["write"]
        current = r["source_hash"] == bench.kernel_source_hash(kernel)
        expect = r["bytes_per_launch"] if current else None
        assert bench.recorded_traffic(kernel, workload) == expect
    assert bench.recorded_traffic("expand", "no_such_workload") is None


def test_layers_per_step_exceed_twice_the_l2():
    l2 = 132_120_576
    for name, shape in W.CONFIGS.items():
        k = bench.layers_per_step(shape, l2)
        assert k >= 4 and k * bench.layer_bytes(shape) > 2 * l2, name


def test_both_arms_describe_the_same_config():
    args = bench.parse_args([])
    assert args.config == "all" and args.steps == 20
    shape = W.CONFIGS[bench.HEADLINE]
    a = bench.config_of(shape, args, 132_120_576, 1)
    assert a["workload"] == "down_proj_graph" and "inputs larger than L2" in a["l2"]
    assert a == bench.config_of(shape, bench.parse_args(["--impl", "reference"]), 132_120_576, 1)
