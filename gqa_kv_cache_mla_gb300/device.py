"""Upload of host workloads (``workloads.py``) to a CUDA device.

Plumbing for the tests and the benchmark: each host array becomes a CUDA
tensor, optionally surrounded by guard bytes filled with a sentinel so a test
can prove that no kernel wrote outside its buffers.  The ``Device*`` classes
hold the tensors of one workload and call the matching entry point of
:mod:`gqa_kv_cache_mla_gb300.kvw`.
"""
from __future__ import annotations

import numpy as np
import torch

from . import kvw
from . import workloads as W

GUARD = 4096
SENTINEL = 0xA5
Q_OUT_FILL = 0xABCD  # bf16 pattern pre-filled in outputs so unwritten rows show

_TORCH_OF = {np.dtype(np.uint8): torch.uint8, np.dtype(np.uint16): torch.int16,
             np.dtype(np.uint32): torch.int32, np.dtype(np.float32): torch.float32,
             np.dtype(np.int32): torch.int32}


class Guarded:
    """A device copy of ``host`` with ``guard`` sentinel bytes on each side."""

    def __init__(self, host: np.ndarray, device, guard: int = GUARD):
        host = np.ascontiguousarray(host)
        self.shape, self.np_dtype, self.guard = host.shape, host.dtype, guard
        n = host.nbytes
        self.raw = torch.full((n + 2 * guard,), SENTINEL, dtype=torch.uint8, device=device)
        if n:
            src = torch.from_numpy(host.reshape(-1).view(np.uint8))
            self.raw[guard:guard + n].copy_(src)
        self.tensor = self.raw[guard:guard + n].view(_TORCH_OF[host.dtype]).view(host.shape)

    def guards_intact(self) -> bool:
        g = self.guard
        if g == 0:
            return True
        return bool((self.raw[:g] == SENTINEL).all()) and bool((self.raw[-g:] == SENTINEL).all())

    def host(self) -> np.ndarray:
        n = int(np.prod(self.shape)) * self.np_dtype.itemsize
        b = self.raw[self.guard:self.guard + n].cpu().numpy()
        return b.view(self.np_dtype).reshape(self.shape)

    def reset(self, host: np.ndarray):
        n = host.nbytes
        if n:
            self.raw[self.guard:self.guard + n].copy_(
                torch.from_numpy(np.ascontiguousarray(host).reshape(-1).view(np.uint8)))


def _cache_desc(c: W.PagedCache, data: Guarded, table: Guarded, lens: Guarded):
    return kvw.paged_cache(data.tensor, c.dtype, table.tensor, lens.tensor, c.num_pages,
                           c.num_layers, c.page_size, c.num_heads, c.head_size, c.strides,
                           scale=c.scale, max_pages_per_seq=c.max_pages_per_seq)


class _Base:
    def _g(self, a, guard):
        g = Guarded(a, self.device, GUARD if guard else 0)
        self.buffers.append(g)
        return g

    def guards_intact(self) -> bool:
        return all(b.guards_intact() for b in self.buffers)

    def flags(self) -> int:
        return int(self.err.host()[0])

    def clear_flags(self):
        self.err.tensor.zero_()


class DeviceMLA(_Base):
    def __init__(self, w: W.MLAWorkload, device="cuda", guard=True, q_out_fill=Q_OUT_FILL):
        self.w, self.device, self.buffers = w, device, []
        c = w.cache
        self.q = self._g(w.q_rope, guard)
        if w.q_out_dtype == W.DTYPE_BF16:
            self.q_out_init = np.full(w.q_rope.shape, q_out_fill, np.uint16)
        else:
            self.q_out_init = np.full(w.q_rope.shape, q_out_fill & 0xFF, np.uint8)
        self.q_out = self._g(self.q_out_init, guard)
        self.kv = self._g(w.kv_in, guard)
        self.offsets = self._g(w.offsets, guard)
        self.freqs = self._g(w.freqs, guard)
        self.gamma = self._g(w.gamma, guard)
        self.cache = self._g(c.data, guard)
        self.page_table = self._g(c.page_table, guard)
        self.cache_lengths = self._g(c.cache_lengths, guard)
        self.err = self._g(np.zeros(1, np.uint32), guard)
        self.desc = _cache_desc(c, self.cache, self.page_table, self.cache_lengths)

    def run(self, stream=None, check=True, **kw):
        w = self.w
        kw.setdefault("num_heads", w.q_rope.shape[1])
        kw.setdefault("tot_seq_len", w.T)
        kw.setdefault("out_dtype", w.q_out_dtype)
        if w.inplace:
            return kvw.kvw_mla_rope_rmsnorm_inplace(
                self.q_out.tensor, self.q.tensor, self.offsets.tensor, self.freqs.tensor,
                self.gamma.tensor, self.desc, w.layer_idx, w.epsilon, self.err.tensor, stream,
                check=check, **kw)
        kw.setdefault("kv_row_stride", w.kv_in.shape[-1])
        return kvw.kvw_mla_rope_rmsnorm_quant(
            self.q_out.tensor, self.q.tensor, self.offsets.tensor, self.freqs.tensor,
            self.gamma.tensor, self.kv.tensor, self.desc, w.layer_idx, w.epsilon,
            self.err.tensor, stream, check=check, **kw)


class DeviceGQA(_Base):
    def __init__(self, w: W.GQAWorkload, device="cuda", guard=True, alias_output=False):
        self.w, self.device, self.buffers = w, device, []
        c = w.cache
        self.q = self._g(w.q_proj, guard)
        self.out_init = np.full(w.q_proj.shape, Q_OUT_FILL, np.uint16)
        self.out = self.q if alias_output else self._g(self.out_init, guard)
        self.offsets = self._g(w.offsets, guard)
        self.freqs = self._g(w.freqs, guard)
        self.pos = None if w.position_ids is None else self._g(w.position_ids, guard)
        self.cache = self._g(c.data, guard)
        self.page_table = self._g(c.page_table, guard)
        self.cache_lengths = self._g(c.cache_lengths, guard)
        self.err = self._g(np.zeros(1, np.uint32), guard)
        self.desc = _cache_desc(c, self.cache, self.page_table, self.cache_lengths)

    def run(self, stream=None, check=True, **kw):
        w = self.w
        kw.setdefault("tot_seq_len", w.T)
        kw.setdefault("num_q_heads", w.q_proj.shape[1])
        return kvw.kvw_qk_rope_paged_ragged(
            self.q.tensor, self.offsets.tensor, self.desc, self.freqs.tensor,
            None if self.pos is None else self.pos.tensor, w.interleaved,
            None if w.mrope_section is None else [int(v) for v in w.mrope_section],
            w.layer_idx, self.out.tensor, self.err.tensor, stream, check=check, **kw)


class DeviceKNorm(_Base):
    def __init__(self, w: W.KNormWorkload, device="cuda", guard=True):
        self.w, self.device, self.buffers = w, device, []
        c = w.cache
        self.offsets = self._g(w.offsets, guard)
        self.gamma = self._g(w.gamma, guard)
        self.cache = self._g(c.data, guard)
        self.page_table = self._g(c.page_table, guard)
        self.cache_lengths = self._g(c.cache_lengths, guard)
        self.err = self._g(np.zeros(1, np.uint32), guard)
        self.desc = _cache_desc(c, self.cache, self.page_table, self.cache_lengths)

    def run(self, stream=None, check=True, per_head_norm=None, **kw):
        w = self.w
        if per_head_norm is None:
            per_head_norm = w.per_head_norm
        return kvw.kvw_rms_norm_kv_cache_paged(
            self.desc, self.gamma.tensor, w.epsilon, w.weight_offset, w.layer_idx, w.T,
            self.offsets.tensor, w.multiply_before_cast, per_head_norm, self.err.tensor, stream,
            check=check, **kw)


class DeviceGather(_Base):
    def __init__(self, w: W.GatherWorkload, device="cuda", guard=True):
        self.w, self.device, self.buffers = w, device, []
        c = w.cache
        self.cache = self._g(c.data, guard)
        self.page_table = self._g(c.page_table, guard)
        self.cache_lengths = self._g(c.cache_lengths, guard)
        self.ctx = self._g(w.ctx_offsets, guard)
        self.out_init = np.zeros((w.rows, 576), np.uint16 if w.out_dtype == W.DTYPE_BF16
                                 else np.uint8)
        self.out = self._g(self.out_init, guard)
        self.scales = self._g(np.zeros(w.rows, np.float32), guard)
        self.err = self._g(np.zeros(1, np.uint32), guard)
        self.desc = _cache_desc(c, self.cache, self.page_table, self.cache_lengths)

    def run(self, stream=None, check=True):
        w = self.w
        if w.dynamic:
            return kvw.kvw_mla_gather_latent_fp8_dynamic(
                self.out.tensor, self.scales.tensor, self.desc, w.layer_idx, self.ctx.tensor,
                self.err.tensor, stream, total_rows=w.rows, check=check)
        return kvw.kvw_mla_gather_latent(self.out.tensor, w.out_dtype, w.out_scale, self.desc,
                                         w.layer_idx, self.ctx.tensor, self.err.tensor, stream,
                                         total_rows=w.rows, check=check)


class DeviceConvert(_Base):
    def __init__(self, w: W.ConvertWorkload, device="cuda", guard=True):
        self.w, self.device, self.buffers = w, device, []
        self.x = self._g(w.x, guard)
        self.out = self._g(np.zeros(w.x.shape, np.uint8), guard)
        self.scales = self._g(np.zeros(w.x.shape[0] if w.per_row else 1, np.float32), guard)
        self.err = self._g(np.zeros(1, np.uint32), guard)  # unused: no data errors here

    def run(self, stream=None, check=True):
        w = self.w
        if w.per_row:
            return kvw.kvw_quantize_fp8_rows(self.out.tensor, self.scales.tensor, self.x.tensor,
                                             stream, check=check)
        return kvw.kvw_convert_bf16_to_fp8_e4m3(self.out.tensor, self.x.tensor, w.scale, stream,
                                                check=check)


def for_workload(w, device="cuda", guard=True):
    """The Device* holder matching the type of workload ``w``."""
    cls = {W.MLAWorkload: DeviceMLA, W.GQAWorkload: DeviceGQA, W.KNormWorkload: DeviceKNorm,
           W.GatherWorkload: DeviceGather, W.ConvertWorkload: DeviceConvert}[type(w)]
    return cls(w, device=device, guard=guard)
