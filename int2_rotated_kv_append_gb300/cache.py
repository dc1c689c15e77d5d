"""Device-side paged caches driven through the C ABI.

``Int2Cache`` owns the INT2 code pool, the fp16 scale/zero pool and the BF16
sink/window buffers of a workload; ``Bf16Cache`` owns the all-BF16 pool of the
speedup reference.  Both only allocate torch memory and call the library, as does
``calibrate`` (the offline step that produces R and the clipping thresholds).
"""

from __future__ import annotations

import torch

from . import (make_dims, oscar_append, oscar_append_mixed, oscar_bf16_append, oscar_bf16_decode, oscar_bf16_decode_workspace_bytes,
               oscar_calibrate, oscar_calibrate_workspace_bytes, oscar_decode, oscar_decode_workspace_bytes,
               oscar_extend, oscar_extend_varlen, oscar_extend_varlen_workspace_bytes, oscar_extend_workspace_bytes)
from .synth import Workload

SENTINEL = 0xA5


class Int2Cache:
    def __init__(self, w: Workload, device="cuda", pages_per_split: int | None = None, fill: int = SENTINEL):
        self.w = w
        self.device = torch.device(device)
        H, D, P, G = w.num_kv_heads, w.head_dim, w.page_size, w.group_size
        self.dims = w.dims
        self.int2_pages = torch.full((w.num_pages * H * 2 * P * D // 4,), fill, dtype=torch.uint8,
                                     device=self.device)
        fill16 = fill * 0x101
        fill16 = fill16 - 0x10000 if fill16 >= 0x8000 else fill16
        self.scale_zero = torch.full((w.num_pages * H * 2 * P * (D // G) * 2,), fill16, dtype=torch.int16,
                                     device=self.device).view(torch.float16)
        self.page_table = w.page_table.to(self.device)
        self.seq_lens = w.seq_lens.to(self.device)
        self.R_k, self.R_v = w.R_k.to(self.device), w.R_v.to(self.device)
        self.clip_k, self.clip_v = w.clip_k.to(self.device), w.clip_v.to(self.device)
        self.offset_k = None if w.offset_k is None else w.offset_k.to(self.device).contiguous()
        self.pps = w.pages_per_split if pages_per_split is None else pages_per_split
        self.sink = None
        self.window = None
        self._ws = None

    def append(self, k, v, slot_mapping, stream=None):
        oscar_append(self.dims, k, v, self.R_k, self.R_v, self.clip_k, self.clip_v, self.page_table, slot_mapping,
                     self.int2_pages, self.scale_zero, stream, offset_k=self.offset_k)

    def prefill(self, stream=None):
        """Append every token of the workload and fill the BF16 sink/window buffers
        (with a key offset, both in one oscar_append_mixed call, which stores the
        offset keys in the BF16 rows)."""
        w = self.w
        if self.offset_k is not None:
            B, H, D = w.batch, w.num_kv_heads, w.head_dim
            self.sink = torch.zeros((B, 2, H, max(w.sink_len, 1), D), dtype=torch.bfloat16, device=self.device)
            self.window = torch.zeros((B, 2, H, max(w.window_len, 1), D), dtype=torch.bfloat16, device=self.device)
            d = self.device
            oscar_append_mixed(self.dims, w.k.to(d), w.v.to(d), self.R_k, self.R_v, self.clip_k, self.clip_v,
                               self.page_table, w.slot_mapping.to(d), w.tok_seq.to(d), w.tok_pos.to(d), self.seq_lens,
                               w.sink_len, w.window_len, self.int2_pages, self.scale_zero, self.sink, self.window,
                               stream, offset_k=self.offset_k)
            return
        self.append(w.k.to(self.device), w.v.to(self.device), w.slot_mapping.to(self.device), stream)
        sink, win = w.sink_window()
        self.sink, self.window = sink.to(self.device), win.to(self.device)

    def workspace(self, max_seq_len=None):
        w = self.w
        msl = w.max_seq_len if max_seq_len is None else max_seq_len
        nbytes = oscar_decode_workspace_bytes(self.dims, w.batch, msl, self.pps, w.sink_len, w.window_len)
        if nbytes == 0:
            raise ValueError("invalid decode arguments for workspace sizing")
        if self._ws is None or self._ws.numel() < nbytes:
            self._ws = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        return self._ws

    def decode(self, q, out=None, sm_scale=0.0, seq_lens=None, max_seq_len=None, stream=None):
        w = self.w
        msl = w.max_seq_len if max_seq_len is None else max_seq_len
        if out is None:
            out = torch.empty((w.batch, w.num_q_heads, w.head_dim), dtype=torch.float32, device=self.device)
        ws = self.workspace(msl)
        oscar_decode(self.dims, w.batch, msl, self.pps, q, self.R_k, self.R_v, self.int2_pages, self.scale_zero,
                     self.sink, self.window, self.page_table, self.seq_lens if seq_lens is None else seq_lens,
                     w.sink_len, w.window_len, sm_scale, out, ws, stream)
        return out


    def extend(self, q, row_seq, row_pos, out=None, sm_scale=0.0, max_seq_len=None, stream=None):
        """Causal attention of query rows q [rows][Hq][D]; row r belongs to sequence
        row_seq[r] at position row_pos[r] (int32 device tensors)."""
        w = self.w
        msl = w.max_seq_len if max_seq_len is None else max_seq_len
        rows = q.shape[0]
        if out is None:
            out = torch.empty((rows, w.num_q_heads, w.head_dim), dtype=torch.float32, device=self.device)
        nbytes = oscar_extend_workspace_bytes(self.dims, rows, msl, self.pps, w.sink_len, w.window_len)
        if nbytes == 0:
            raise ValueError("invalid extend arguments for workspace sizing")
        if self._ws is None or self._ws.numel() < nbytes:
            self._ws = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        oscar_extend(self.dims, w.batch, msl, self.pps, q, row_seq, row_pos, self.R_k, self.R_v, self.int2_pages,
                     self.scale_zero, self.sink, self.window, self.page_table, self.seq_lens, w.sink_len,
                     w.window_len, sm_scale, out, self._ws, stream)
        return out


    def extend_varlen(self, q, q_start, max_rows_per_seq, out=None, sm_scale=0.0, max_seq_len=None, stream=None):
        """Causal attention of the rows q [rows][Hq][D], rows q_start[b] .. q_start[b+1]-1
        being the last positions of sequence b (int32 device q_start [B+1])."""
        w = self.w
        msl = w.max_seq_len if max_seq_len is None else max_seq_len
        rows = q.shape[0]
        if out is None:
            out = torch.empty((rows, w.num_q_heads, w.head_dim), dtype=torch.float32, device=self.device)
        nbytes = oscar_extend_varlen_workspace_bytes(self.dims, rows, msl, self.pps, w.sink_len, w.window_len)
        if nbytes == 0:
            raise ValueError("invalid extend arguments for workspace sizing")
        if self._ws is None or self._ws.numel() < nbytes:
            self._ws = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        oscar_extend_varlen(self.dims, w.batch, msl, max_rows_per_seq, self.pps, q, q_start, self.R_k, self.R_v,
                            self.int2_pages, self.scale_zero, self.sink, self.window, self.page_table, self.seq_lens,
                            w.sink_len, w.window_len, sm_scale, out, self._ws, stream)
        return out


class Bf16Cache:
    def __init__(self, w: Workload, device="cuda", pages_per_split: int | None = None):
        self.w = w
        self.device = torch.device(device)
        self.dims = w.dims
        self.pages = torch.zeros((w.num_pages * w.num_kv_heads * 2 * w.page_size * w.head_dim,),
                                 dtype=torch.bfloat16, device=self.device)
        self.page_table = w.page_table.to(self.device)
        self.seq_lens = w.seq_lens.to(self.device)
        self.pps = w.pages_per_split if pages_per_split is None else pages_per_split
        self._ws = None

    def prefill(self, stream=None):
        w = self.w
        oscar_bf16_append(self.dims, w.k.to(self.device), w.v.to(self.device), w.slot_mapping.to(self.device),
                          self.pages, stream)

    def workspace(self):
        w = self.w
        nbytes = oscar_bf16_decode_workspace_bytes(self.dims, w.batch, w.max_seq_len, self.pps)
        if self._ws is None or self._ws.numel() < nbytes:
            self._ws = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        return self._ws

    def decode(self, q, out=None, sm_scale=0.0, stream=None):
        w = self.w
        if out is None:
            out = torch.empty((w.batch, w.num_q_heads, w.head_dim), dtype=torch.float32, device=self.device)
        oscar_bf16_decode(self.dims, w.batch, w.max_seq_len, self.pps, q, self.pages, self.page_table,
                          self.seq_lens, sm_scale, out, self.workspace(), stream)
        return out


def calibrate(k=None, v=None, centered: bool = True, clip_quantile: float = 1.0, with_cov: bool = False,
              workspace=None, stream=None) -> dict:
    """R, clipping thresholds and eigenvalues per KV head from calibration samples
    (device bf16 [N][Hkv][D]); returns {"k": {...}, "v": {...}} for the sides given,
    each with R [Hkv][D][D], clip [Hkv][D], eigenvalues [Hkv][D], sweeps [Hkv] and,
    with ``with_cov``, cov [Hkv][D][D]."""
    x = k if k is not None else v
    if x is None:
        raise ValueError("calibrate needs k or v samples")
    N, H, D = x.shape
    dims = make_dims(H, H, D, 16, D, 1, 1)
    dev = x.device

    def outputs():
        o = {"R": torch.empty(H, D, D, dtype=torch.float32, device=dev),
             "clip": torch.empty(H, D, dtype=torch.float32, device=dev),
             "eigenvalues": torch.empty(H, D, dtype=torch.float32, device=dev),
             "sweeps": torch.empty(H, dtype=torch.int32, device=dev)}
        if with_cov:
            o["cov"] = torch.empty(H, D, D, dtype=torch.float32, device=dev)
        return o

    out_k = outputs() if k is not None else None
    out_v = outputs() if v is not None else None
    if workspace is None:
        workspace = torch.empty(oscar_calibrate_workspace_bytes(dims, N), dtype=torch.uint8, device=dev)
    oscar_calibrate(dims, N, k, v, int(centered), clip_quantile, out_k, out_v, workspace, stream)
    res = {}
    if out_k is not None:
        res["k"] = out_k
    if out_v is not None:
        res["v"] = out_v
    return res
