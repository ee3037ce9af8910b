"""Shared helpers for the GPU parity tests: moving seeded inputs to the device,
guarded buffers, running the library path and the oracle, tolerance checks."""
from __future__ import annotations

import numpy as np

import oracle
from gathered_rank_gemm_gb300 import binding
from gathered_rank_gemm_gb300 import workloads as W

U_SENTINEL_BITS = 0x7FC0DEAD   # fp32 NaN pattern pre-filled in u
GUARD_BYTES = 256
RTOL = 1e-2
ATOL = 1e-2


def torch_mod():
    import torch
    return torch


def bf16_dev(a: np.ndarray, dev):
    torch = torch_mod()
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)


def f16_dev(a: np.ndarray, dev):
    torch = torch_mod()
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.float16)


def bits_of(t) -> np.ndarray:
    torch = torch_mod()
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


class Guarded:
    """A device buffer with sentinel-filled guard bands before and after."""

    def __init__(self, shape, dtype, dev, fill_bits: int | None = None, init=None):
        torch = torch_mod()
        self.dtype = dtype
        esz = torch.empty((), dtype=dtype).element_size()
        self.g = GUARD_BYTES // esz
        numel = int(np.prod(shape))
        self.full = torch.empty(numel + 2 * self.g, dtype=dtype, device=dev)
        int_dt = {1: torch.uint8, 2: torch.int16, 4: torch.int32, 8: torch.int64}[esz]
        self.full.view(int_dt).fill_(0x5A5A if esz == 2 else 0x5A)
        if esz == 4:
            self.full.view(torch.int32).fill_(0x5A5A5A5A)
        self.view = self.full[self.g:self.g + numel].view(*shape)
        if fill_bits is not None:
            self.view.view(int_dt).fill_(fill_bits - (1 << (8 * esz)) if fill_bits >= 1 << (8 * esz - 1) else fill_bits)
        if init is not None:
            self.view.copy_(init)
        self._int_dt = int_dt
        self.guard_before = self.full[:self.g].view(int_dt).clone()
        self.guard_after = self.full[self.g + numel:].view(int_dt).clone()

    def guards_intact(self) -> bool:
        torch = torch_mod()
        numel = self.view.numel()
        a = torch.equal(self.full[:self.g].view(self._int_dt), self.guard_before)
        b = torch.equal(self.full[self.g + numel:].view(self._int_dt), self.guard_after)
        return bool(a and b)


class DeviceCase:
    """One layer's inputs on the device plus the metadata buffers (guarded)."""

    def __init__(self, shape: W.LayerShape, mapping: np.ndarray, layer: W.Layer, dev,
                 x_pad: int = 0, y_pad: int = 0, split_workspace: bool = False,
                 lora_scales=None, paged: bool = False, f16: bool = False):
        torch = torch_mod()
        # fp16 inputs: the same draws rounded to fp16, through the *_f16 entry points
        self.f16 = f16
        if f16:
            assert not paged, "paged weights are bf16 only"
            layer = W.layer_as_f16(layer)
        dev16 = f16_dev if f16 else bf16_dev
        dt16 = torch.float16 if f16 else torch.bfloat16
        self.shape, self.mapping_np, self.layer, self.dev = shape, mapping, layer, dev
        # per-adapter factors on the scale (float32 values, also given to the oracle)
        self.lora_scales_np = None if lora_scales is None else np.asarray(lora_scales, np.float32)
        self.lora_scales = (None if lora_scales is None else
                            torch_mod().from_numpy(self.lora_scales_np.copy()).to(dev))
        T, L = shape.max_num_tokens, shape.max_loras
        self.mapping = torch.from_numpy(mapping).to(dev)
        self.n = torch.tensor([shape.num_tokens], dtype=torch.int32, device=dev)
        xs = np.zeros((T, shape.hidden + x_pad), np.uint16)
        xs[:, :shape.hidden] = layer.x
        if x_pad:
            xs[:, shape.hidden:] = W.BF16_QNAN_PAYLOAD   # never read
        self.x_full = dev16(xs, dev)
        self.x = self.x_full[:, :shape.hidden]
        ys = np.zeros((T, shape.out_width + y_pad), np.uint16)
        ys[:, :shape.out_width] = layer.y
        if y_pad:
            ys[:, shape.out_width:] = W.BF16_Y_SENTINEL
        self.y_in_bits = ys
        self.y = Guarded((T, shape.out_width + y_pad), dt16, dev, init=dev16(ys, dev))
        self.y_view = self.y.view[:, :shape.out_width]
        self.a = [dev16(v, dev) for v in layer.lora_a]
        self.b = [dev16(v, dev) for v in layer.lora_b]
        # paged weights: every adapter's A_s[l] / B_s[l] in its own allocation
        # (allocated in reverse adapter order), found through address tables
        self.paged = paged
        if paged:
            torch = torch_mod()
            L_ = shape.max_loras
            self.a_pages = [[None] * L_ for _ in layer.lora_a]
            self.b_pages = [[None] * L_ for _ in layer.lora_b]
            for l in reversed(range(L_)):
                for s_ in range(shape.num_slices):
                    self.a_pages[s_][l] = bf16_dev(layer.lora_a[s_][l], dev)
                    self.b_pages[s_][l] = bf16_dev(layer.lora_b[s_][l], dev)
            self.a_tables = [torch.tensor([t.data_ptr() for t in pages], dtype=torch.int64,
                                          device=dev) for pages in self.a_pages]
            self.b_tables = [torch.tensor([t.data_ptr() for t in pages], dtype=torch.int64,
                                          device=dev) for pages in self.b_pages]
        self.u = Guarded((shape.num_slices, T, shape.rank), torch.float32, dev,
                         fill_bits=U_SENTINEL_BITS)
        self.sorted = Guarded((T,), torch.int32, dev, fill_bits=0x11111111)
        self.counts = Guarded((L + 1,), torch.int32, dev, fill_bits=0x22222222)
        self.starts = Guarded((L + 2,), torch.int32, dev, fill_bits=0x33333333)
        self.ws_base = binding.lora_workspace_size(T, L)
        ws_bytes = self.ws_base
        if split_workspace:
            ws_bytes = binding.lora_shrink_expand_workspace_size(
                T, L, shape.hidden, shape.slice_widths, shape.rank)
        self.ws = Guarded((ws_bytes,), torch.uint8, dev, fill_bits=0)

    def prepare(self, stream=None):
        binding.lora_prepare_metadata(self.mapping, self.n, self.shape.max_loras,
                                      self.sorted.view, self.counts.view, self.starts.view,
                                      self.ws.view, stream)

    def shrink(self, stream=None):
        if self.paged:
            binding.lora_shrink_paged(self.x, self.a_tables, self.shape.rank, self.shape.scale,
                                      self.u.view, self.sorted.view, self.starts.view,
                                      self.ws.view, stream, self.lora_scales)
            return
        binding.lora_shrink(self.x, self.a, self.shape.scale, self.u.view, self.sorted.view,
                            self.starts.view, self.ws.view, stream, self.lora_scales)

    def expand(self, stream=None, u=None):
        if self.paged:
            binding.lora_expand_paged(self.u.view if u is None else u, self.b_tables,
                                      self.shape.slice_widths, self.y_view, self.sorted.view,
                                      self.starts.view, self.ws.view, stream)
            return
        binding.lora_expand(self.u.view if u is None else u, self.b, self.y_view,
                            self.sorted.view, self.starts.view, self.ws.view, stream)

    def shrink_expand(self, stream=None):
        if self.paged:
            binding.lora_shrink_expand_paged(self.x, self.a_tables, self.b_tables,
                                             self.shape.slice_widths, self.shape.scale,
                                             self.u.view, self.y_view, self.sorted.view,
                                             self.starts.view, self.ws.view, stream,
                                             self.lora_scales)
            return
        binding.lora_shrink_expand(self.x, self.a, self.b, self.shape.scale, self.u.view,
                                   self.y_view, self.sorted.view, self.starts.view, self.ws.view,
                                   stream, self.lora_scales)

    def run(self, fused: bool = False):
        self.prepare()
        if fused:
            self.shrink_expand()
        else:
            self.shrink()
            self.expand()
        torch_mod().cuda.synchronize()

    def guards_intact(self):
        return all(g.guards_intact() for g in (self.y, self.u, self.sorted, self.counts,
                                                self.starts, self.ws))


def within_tol(gpu: np.ndarray, ref: np.ndarray):
    """Per-element |gpu - ref| <= 1e-2 + 1e-2 |ref|; returns (ok, worst ratio)."""
    err = np.abs(gpu - ref)
    bound = ATOL + RTOL * np.abs(ref)
    ratio = float(np.max(err / bound)) if err.size else 0.0
    return bool(np.all(err <= bound)), ratio


def lora_rows(mapping: np.ndarray, n: int, L: int) -> np.ndarray:
    m = mapping[:n]
    return np.nonzero((m >= 0) & (m < L))[0]


def check_case(case: DeviceCase, *, full_oracle: bool = True, sample_rows=None,
               fused: bool = False):
    """Runs the path (shrink + expand, or the one-call shrink_expand) and checks
    metadata (bit-exact), u and y (tolerance), untouched rows (bit-exact) and
    guard bands.  Returns diagnostics."""
    sh, lay = case.shape, case.layer
    T, L, n = sh.max_num_tokens, sh.max_loras, sh.num_tokens
    case.run(fused=fused)
    s_ref, c_ref, st_ref, status_ref = oracle.prepare_metadata(case.mapping_np, n, L)
    assert np.array_equal(case.sorted.view.cpu().numpy(), s_ref), "sorted_token_ids differ"
    assert np.array_equal(case.counts.view.cpu().numpy(), c_ref), "num_tokens_per_lora differ"
    assert np.array_equal(case.starts.view.cpu().numpy(), st_ref), "lora_token_start_loc differ"
    assert case.guards_intact(), "a guard band was overwritten"

    rows = lora_rows(case.mapping_np, n, L)
    if sample_rows is not None and len(rows) > sample_rows:
        rows = np.sort(np.random.default_rng(5).choice(rows, sample_rows, replace=False))
    keep = np.zeros(T, bool)
    keep[lora_rows(case.mapping_np, n, L)] = True

    u_gpu = case.u.view.cpu().numpy()
    u_bits = u_gpu.view(np.uint32)
    assert np.all(u_bits[:, ~keep, :] == U_SENTINEL_BITS), "u rows without adapter were written"

    # oracle on the selected rows only (others: mapping -1 so the oracle skips them)
    m_sel = np.full(T, -1, np.int32)
    m_sel[rows] = case.mapping_np[rows]
    u_ref = oracle.shrink(lay.x, lay.lora_a, sh.scale, m_sel, n, L,
                          u_init=np.zeros((sh.num_slices, T, sh.rank)),
                          lora_scales=None if case.lora_scales_np is None
                          else case.lora_scales_np.astype(np.float64), f16=case.f16)
    ok_u, r_u = within_tol(u_gpu[:, rows].astype(np.float64), u_ref[:, rows])
    assert ok_u, f"u differs from the oracle (worst err/bound {r_u:.3f})"

    y_gpu_bits = bits_of(case.y.view)
    y_gpu = oracle.decode_bits(y_gpu_bits, f16=case.f16)
    y_in = case.y_in_bits
    untouched = ~keep
    assert np.array_equal(y_gpu_bits[untouched], y_in[untouched]), "y rows without adapter changed"
    if y_in.shape[1] > sh.out_width:
        assert np.array_equal(y_gpu_bits[:, sh.out_width:], y_in[:, sh.out_width:]), \
            "y columns past the slices changed"
    y_in_used = np.ascontiguousarray(y_in[:, :sh.out_width])
    # (i) end to end: oracle u in fp64
    y_ref = oracle.expand(u_ref, lay.lora_b, y_in_used, m_sel, n, L, f16=case.f16)
    ok_y, r_y = within_tol(y_gpu[rows, :sh.out_width], y_ref[rows])
    assert ok_y, f"y differs from the oracle end to end (worst err/bound {r_y:.3f})"
    # (ii) expand alone: the GPU's own u fed to the oracle, zero base output
    zero_y = np.zeros_like(y_in_used)
    d_ref = oracle.expand(np.nan_to_num(u_gpu.astype(np.float64)), lay.lora_b, zero_y, m_sel, n, L,
                          f16=case.f16)
    d_gpu = y_gpu[rows, :sh.out_width] - oracle.decode_bits(y_in_used[rows], f16=case.f16)
    # the GPU delta carries the final 16-bit rounding of y: bound it by an ulp
    # of y (8 significand bits for bf16, 11 for fp16)
    ulp = np.abs(y_gpu[rows, :sh.out_width]) * 2.0 ** (-10 if case.f16 else -8)
    err = np.abs(d_gpu - d_ref[rows])
    assert np.all(err <= ATOL + RTOL * np.abs(d_ref[rows]) + ulp), \
        "expand delta differs from the oracle's expand of the GPU u"
    return dict(rows=len(rows), worst_u=r_u, worst_y=r_y)
