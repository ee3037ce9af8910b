"""Seeded synthetic inputs for multi-LoRA shrink/expand.

This module only draws inputs: token->LoRA mappings, activations, adapter
weights and base outputs, as numpy arrays (bf16 values are carried as their
uint16 bit patterns).  It holds none of the method's arithmetic, so both the
fp64 oracle and the CUDA library can be fed from it.

The five named workloads stand in for the vLLM serving runs on the pages
(Llama-2-7B, ShareGPT, 4 adapters of rank 8, "[V1] LoRA - Add triton
kernels for V1", benchmark section); the model, dataset and adapters are not
used.  Their recipe:

* ``tiny``            64 tokens, hidden 512, one slice of 512, 4 LoRAs of rank 8,
                      ids uniform over {-1, 0, 1, 2, 3}
* ``decode_qkv``      256 tokens, hidden 4096, three slices of 4096, 4 LoRAs of
                      rank 8, -1 with probability 0.10, else uniform over 0..3
* ``chunked_prefill`` 8192 tokens, hidden 4096, one slice of 4096, 8 LoRAs of
                      rank 16; request runs of geometric length (mean 512), each
                      run one uniform id, runs concatenated in draw order
* ``mlp_gate_up``     2048 tokens, hidden 4096, two slices of 11008, 32 LoRAs of
                      rank 64, -1 with probability 0.05, else Zipf(1.1) over 32 ids
* ``down_proj_graph`` buffer of 8192 tokens with 5000 valid, hidden 11008, one
                      slice of 4096, 128 LoRAs of rank 128, -1 with probability
                      0.25, else uniform; the pad rows t >= 5000 hold garbage:
                      random int32 ids (valid ones included), NaN / huge bf16
                      patterns in x, a sentinel pattern in y

x ~ N(0, 1), A and B ~ N(0, 0.02), base output y ~ N(0, 1), scale 1.0, all
rounded to bf16 with round-to-nearest-even.  Seeds are 1000 + the workload's
index in the list above, plus the layer index for multi-layer benchmarks.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# bf16 bit patterns used as garbage / sentinels in the pad region
BF16_QNAN_PAYLOAD = 0x7FC1      # a quiet NaN with a payload
BF16_HUGE = 0x7F7F              # largest finite bf16 (~3.39e38)
BF16_Y_SENTINEL = 0x7FA5        # NaN pattern left in y rows that must stay untouched


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); finite inputs only."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


@dataclass(frozen=True)
class LayerShape:
    """Sizes of one LoRA-wrapped linear layer and its batch."""
    name: str
    max_num_tokens: int          # T_max: static buffer rows
    num_tokens: int              # n: valid rows (n <= T_max)
    hidden: int                  # H: input width (shrink K)
    slice_widths: tuple          # N_s for each of the S output slices
    max_loras: int               # L
    rank: int                    # R
    scale: float = 1.0
    mapping: str = "uniform"     # recipe name, see make_mapping
    neg_prob: float = 0.0        # probability of -1 (recipes that use it)
    index: int = 0               # position in the named list (seed offset)

    @property
    def num_slices(self) -> int:
        return len(self.slice_widths)

    @property
    def out_width(self) -> int:
        return int(sum(self.slice_widths))


CONFIGS = {
    "tiny": LayerShape("tiny", 64, 64, 512, (512,), 4, 8, 1.0, "uniform_incl_neg", 0.0, 0),
    "decode_qkv": LayerShape("decode_qkv", 256, 256, 4096, (4096, 4096, 4096), 4, 8, 1.0,
                             "uniform", 0.10, 1),
    "chunked_prefill": LayerShape("chunked_prefill", 8192, 8192, 4096, (4096,), 8, 16, 1.0,
                                  "runs", 0.0, 2),
    "mlp_gate_up": LayerShape("mlp_gate_up", 2048, 2048, 4096, (11008, 11008), 32, 64, 1.0,
                              "zipf", 0.05, 3),
    "down_proj_graph": LayerShape("down_proj_graph", 8192, 5000, 11008, (4096,), 128, 128, 1.0,
                                  "uniform", 0.25, 4),
}


def make_mapping(shape: LayerShape, rng: np.random.Generator) -> np.ndarray:
    """token_lora_mapping[T_max] (int32); entries t >= n are pad garbage."""
    n, t_max, nl = shape.num_tokens, shape.max_num_tokens, shape.max_loras
    kind = shape.mapping
    if kind == "uniform_incl_neg":
        valid = rng.integers(-1, nl, size=n)
    elif kind == "uniform":
        valid = rng.integers(0, nl, size=n)
        valid[rng.random(n) < shape.neg_prob] = -1
    elif kind == "zipf":
        k = np.arange(1, nl + 1, dtype=np.float64)
        p = k ** -1.1
        p /= p.sum()
        valid = rng.choice(nl, size=n, p=p)
        valid[rng.random(n) < shape.neg_prob] = -1
    elif kind == "runs":
        parts, total = [], 0
        while total < n:
            length = int(rng.geometric(1.0 / 512.0))
            length = min(length, n - total)
            parts.append(np.full(length, rng.integers(0, nl), dtype=np.int64))
            total += length
        valid = np.concatenate(parts)
    elif kind == "all_zero":
        valid = np.zeros(n, np.int64)
    else:
        raise ValueError(f"unknown mapping recipe {kind!r}")
    m = np.empty(t_max, np.int32)
    m[:n] = valid
    if t_max > n:
        # pad garbage: arbitrary int32, with valid ids mixed in on purpose
        tail = rng.integers(-2**31, 2**31 - 1, size=t_max - n, dtype=np.int64)
        pick = rng.random(t_max - n) < 0.5
        tail[pick] = rng.integers(-1, nl, size=int(pick.sum()))
        m[n:] = tail.astype(np.int32)
    return m


def _normal_bf16(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return f32_to_bf16_bits(a)


@dataclass
class Layer:
    """One layer instance: activations, adapter weights and base output."""
    x: np.ndarray                # uint16 [T_max, H]
    lora_a: list                 # S x uint16 [L, R, H]
    lora_b: list                 # S x uint16 [L, R, N_s]
    y: np.ndarray                # uint16 [T_max, sum N_s]


@dataclass
class Workload:
    shape: LayerShape
    mapping: np.ndarray          # int32 [T_max]
    layers: list = field(default_factory=list)


def make_layer(shape: LayerShape, rng: np.random.Generator, *, garbage_tail: bool = True) -> Layer:
    t_max, n, h = shape.max_num_tokens, shape.num_tokens, shape.hidden
    x = _normal_bf16(rng, (t_max, h), 1.0)
    y = _normal_bf16(rng, (t_max, shape.out_width), 1.0)
    if garbage_tail and t_max > n:
        x[n:] = np.where((np.arange(h) % 2) == 0, BF16_QNAN_PAYLOAD, BF16_HUGE).astype(np.uint16)
        y[n:] = BF16_Y_SENTINEL
    lora_a = [_normal_bf16(rng, (shape.max_loras, shape.rank, h), 0.02)
              for _ in range(shape.num_slices)]
    lora_b = [_normal_bf16(rng, (shape.max_loras, shape.rank, w), 0.02)
              for w in shape.slice_widths]
    return Layer(x=x, lora_a=lora_a, lora_b=lora_b, y=y)


def make_workload(shape: LayerShape | str, num_layers: int = 1, seed: int | None = None) -> Workload:
    """The mapping plus ``num_layers`` independent layer instances."""
    if isinstance(shape, str):
        shape = CONFIGS[shape]
    base = 1000 + shape.index if seed is None else seed
    rng = np.random.default_rng(base)
    wl = Workload(shape=shape, mapping=make_mapping(shape, rng))
    for k in range(num_layers):
        wl.layers.append(make_layer(shape, np.random.default_rng([base, k])))
    return wl


def custom_shape(name: str = "custom", *, max_num_tokens: int, num_tokens: int | None = None,
                 hidden: int, slice_widths, max_loras: int, rank: int, scale: float = 1.0,
                 mapping: str = "uniform", neg_prob: float = 0.1) -> LayerShape:
    """A LayerShape for tests (same recipes as the named workloads)."""
    return LayerShape(name, max_num_tokens, max_num_tokens if num_tokens is None else num_tokens,
                      hidden, tuple(slice_widths), max_loras, rank, scale, mapping, neg_prob, 0)


def to_f16_bits(bits: np.ndarray) -> np.ndarray:
    """The values of bf16 bit patterns rounded to IEEE fp16 (numpy's float16
    cast: nearest, ties to even; out-of-range values become infinities)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    with np.errstate(over="ignore", invalid="ignore"):
        f = (b.astype(np.uint32) << 16).view(np.float32).astype(np.float16)
    return f.view(np.uint16)


def layer_as_f16(layer: Layer) -> Layer:
    """The same layer drawn in fp16: every input array's values as fp16 bits
    (the pad-row NaN / huge garbage stays NaN / becomes infinity)."""
    return Layer(x=to_f16_bits(layer.x), lora_a=[to_f16_bits(a) for a in layer.lora_a],
                 lora_b=[to_f16_bits(b) for b in layer.lora_b], y=to_f16_bits(layer.y))
