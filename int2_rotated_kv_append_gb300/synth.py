"""Seeded synthetic workloads for the OSCAR append/decode path.

This module only draws inputs: token K/V vectors, queries, orthogonal
rotations, clip thresholds, page tables, slot mappings and sequence lengths.
It holds none of the method's arithmetic (no quantisation, no attention), so
the CUDA path and the CPU oracle can both be fed from it.

The shapes and value distributions follow the workloads the OSCAR pages
evaluate (Qwen3-class models: 32 query / 8 KV heads of dimension 128, long
reasoning traces and contexts up to 128K; "OSCAR: Offline Spectral
Covariance-Aware Rotation for 2-bit KV Cache Quantization", abstract).  No
model, dataset or benchmark item is used.

Draw recipe (fixed order, seed = config index unless given):
  * small draws (rotations, channel means, outlier channels, page tables,
    lengths, slots) come from a CPU ``torch.Generator`` and are therefore the
    same on every device;
  * bulk draws (K, V, q) come from a generator on the target device, in fp32,
    rounded to bf16 with round-to-nearest-even;
  * rotations are Haar-random: QR of a Gaussian fp64 matrix with the signs of
    R's diagonal folded into Q, then stored as fp32;
  * clip thresholds are synthetic stand-ins for the offline calibration:
    0.9 x the per-channel max |x . R| over all tokens of that head, computed
    with a library fp64 matmul and stored as fp32.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

PAGE_SIZE = 16


@dataclasses.dataclass
class Workload:
    """One synthetic problem: cache contents, queries and layout metadata."""

    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    group_size: int
    sink_len: int
    window_len: int
    batch: int
    num_pages: int
    max_pages_per_seq: int
    pages_per_split: int
    seq_lens: torch.Tensor          # int32 [B] (cpu)
    page_table: torch.Tensor        # int32 [B][max_pages_per_seq] (cpu), -1 = unused
    k: torch.Tensor                 # bf16 [T][Hkv][D] every token of every sequence, in order
    v: torch.Tensor                 # bf16 [T][Hkv][D]
    tok_seq: torch.Tensor           # int32 [T] sequence of each token (cpu)
    tok_pos: torch.Tensor           # int32 [T] position of each token (cpu)
    slot_mapping: torch.Tensor      # int64 [T] page * P + offset (cpu)
    q: torch.Tensor                 # bf16 [B][Hq][D]
    R_k: torch.Tensor               # fp32 [Hkv][D][D]
    R_v: torch.Tensor               # fp32 [Hkv][D][D]
    clip_k: torch.Tensor            # fp32 [Hkv][D]
    clip_v: torch.Tensor            # fp32 [Hkv][D]
    seed: int = 0
    offset_k: torch.Tensor | None = None  # fp32 [Hkv][D] key offset (None: keys are not offset)

    @property
    def dims(self) -> dict:
        return dict(num_q_heads=self.num_q_heads, num_kv_heads=self.num_kv_heads, head_dim=self.head_dim,
                    page_size=self.page_size, group_size=self.group_size, num_pages=self.num_pages,
                    max_pages_per_seq=self.max_pages_per_seq)

    @property
    def num_tokens(self) -> int:
        return int(self.k.shape[0])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max().item()) if self.batch else 0

    def sink_window(self) -> tuple[torch.Tensor, torch.Tensor]:
        """BF16 sink [B][2][Hkv][S][D] and window ring [B][2][Hkv][W][D] holding the
        original (unrotated) K/V of positions p < S and of p in [max(S, L-W), L)
        at ring slot p % W.  Slots that hold no token are zero.  Workloads with a key
        offset have no such buffers here: the library's mixed append writes them."""
        if self.offset_k is not None:
            raise ValueError("sink/window of a workload with a key offset come from oscar_append_mixed")
        B, H, D, S, W = self.batch, self.num_kv_heads, self.head_dim, self.sink_len, self.window_len
        dev = self.k.device
        sink = torch.zeros((B, 2, H, max(S, 1), D), dtype=torch.bfloat16, device=dev)
        win = torch.zeros((B, 2, H, max(W, 1), D), dtype=torch.bfloat16, device=dev)
        seq = self.tok_seq.to(torch.int64)
        pos = self.tok_pos.to(torch.int64)
        L = self.seq_lens.to(torch.int64)[seq]
        in_sink = pos < S
        win_begin = torch.clamp(L - W, min=S)
        in_win = (pos >= win_begin) & (pos < L) & (W > 0)
        idx = torch.nonzero(in_sink).flatten()
        if idx.numel():
            i_d = idx.to(dev)
            sink[seq[idx].to(dev), 0, :, pos[idx].to(dev)] = self.k[i_d]
            sink[seq[idx].to(dev), 1, :, pos[idx].to(dev)] = self.v[i_d]
        idx = torch.nonzero(in_win).flatten()
        if idx.numel():
            i_d = idx.to(dev)
            slot = (pos[idx] % max(W, 1)).to(dev)
            win[seq[idx].to(dev), 0, :, slot] = self.k[i_d]
            win[seq[idx].to(dev), 1, :, slot] = self.v[i_d]
        return sink, win


def haar_orthogonal(n: int, D: int, gen: torch.Generator) -> torch.Tensor:
    """n Haar-random orthogonal D x D matrices, fp64 (cpu)."""
    g = torch.randn((n, D, D), dtype=torch.float64, generator=gen)
    qm, rm = torch.linalg.qr(g)
    sign = torch.sign(torch.diagonal(rm, dim1=-2, dim2=-1))
    sign[sign == 0] = 1.0
    return qm * sign.unsqueeze(-2)


def clip_thresholds(x: torch.Tensor, R: torch.Tensor, frac: float = 0.9, chunk: int = 65536) -> torch.Tensor:
    """frac x per-channel max |x . R| over all tokens (x bf16 [T][H][D], R fp32 [H][D][D])."""
    T, H, D = x.shape
    out = torch.zeros((H, D), dtype=torch.float64, device=x.device)
    Rd = R.to(x.device, torch.float64)
    for h in range(H):
        for t0 in range(0, T, chunk):
            xr = x[t0:t0 + chunk, h].to(torch.float64) @ Rd[h]
            out[h] = torch.maximum(out[h], xr.abs().amax(dim=0))
    return (frac * out).to(torch.float32).cpu()


def _draw_k(T: int, H: int, D: int, gen_cpu, gen_dev, device, kind: str) -> torch.Tensor:
    """K vectors.  kind 'tiny': N(0,1) with 4 outlier channels x20 per head.
    kind 'qwen': per-head channel means ~N(0, 3^2) plus unit noise, with 6 outlier
    channels per head (drawn without replacement) whose whole value x15."""
    noise = torch.randn((T, H, D), dtype=torch.float32, generator=gen_dev, device=device)
    scale = torch.ones((H, D), dtype=torch.float32)
    if kind == "tiny":
        mean = torch.zeros((H, D), dtype=torch.float32)
        n_out, factor = 4, 20.0
    else:
        mean = 3.0 * torch.randn((H, D), dtype=torch.float32, generator=gen_cpu)
        n_out, factor = 6, 15.0
    for h in range(H):
        ch = torch.randperm(D, generator=gen_cpu)[:n_out]
        scale[h, ch] = factor
    x = (noise + mean.to(device)) * scale.to(device)
    return x.to(torch.bfloat16)


def _normal_bf16(shape, gen_dev, device) -> torch.Tensor:
    return torch.randn(shape, dtype=torch.float32, generator=gen_dev, device=device).to(torch.bfloat16)


def make_workload(*, num_q_heads: int, num_kv_heads: int, head_dim: int, group_size: int, sink_len: int,
                  window_len: int, seq_lens, seed: int, device="cpu", k_kind: str = "qwen",
                  page_size: int = PAGE_SIZE, pages_per_split: int = 0, spare_pages: int = 0,
                  shuffle_pages: bool = True, name: str = "custom", same_rotation: bool = False,
                  clip_frac: float | None = 0.9, key_offset: bool = False) -> Workload:
    """Build a workload with the given shape.  Every sequence's tokens are drawn
    and given slots in a shared page pool (random page order when shuffled).
    ``key_offset``: the workload carries a key offset, the per-(KV head, channel)
    mean of its keys in fp32, and K's clipping thresholds are taken on k - offset."""
    device = torch.device(device)
    gen_cpu = torch.Generator(device="cpu").manual_seed(seed)
    gen_dev = torch.Generator(device=device).manual_seed(seed + 1_000_003)
    seq_lens = [int(x) for x in seq_lens]
    B = len(seq_lens)
    H, Hq, D, P = num_kv_heads, num_q_heads, head_dim, page_size
    pages_per_seq = [max(1, math.ceil(L / P)) for L in seq_lens]
    max_pages = max(pages_per_seq) if B else 1
    num_pages = sum(pages_per_seq) + spare_pages
    order = torch.randperm(num_pages, generator=gen_cpu) if shuffle_pages else torch.arange(num_pages)
    page_table = torch.full((B, max_pages), -1, dtype=torch.int32)
    cursor = 0
    for b, n in enumerate(pages_per_seq):
        page_table[b, :n] = order[cursor:cursor + n].to(torch.int32)
        cursor += n
    rots = haar_orthogonal(2 * H, D, gen_cpu)
    R_k = rots[:H].to(torch.float32).contiguous()
    R_v = R_k.clone() if same_rotation else rots[H:].to(torch.float32).contiguous()
    T = sum(seq_lens)
    k = _draw_k(T, H, D, gen_cpu, gen_dev, device, k_kind)
    v = _normal_bf16((T, H, D), gen_dev, device)
    q = _normal_bf16((B, Hq, D), gen_dev, device)
    tok_seq = torch.cat([torch.full((L,), b, dtype=torch.int32) for b, L in enumerate(seq_lens)]) if T else \
        torch.zeros(0, dtype=torch.int32)
    tok_pos = torch.cat([torch.arange(L, dtype=torch.int32) for L in seq_lens]) if T else \
        torch.zeros(0, dtype=torch.int32)
    pages = page_table.to(torch.int64)[tok_seq.to(torch.int64), (tok_pos // P).to(torch.int64)]
    slot_mapping = pages * P + (tok_pos % P).to(torch.int64)
    offset_k = k.to(torch.float32).mean(dim=0).contiguous() if key_offset and T else None
    if clip_frac is None:
        clip_k = torch.full((H, D), float("inf"), dtype=torch.float32)
        clip_v = clip_k.clone()
    else:
        clip_k = clip_thresholds(k if offset_k is None else k.to(torch.float32) - offset_k, R_k, clip_frac)
        clip_v = clip_thresholds(v, R_v, clip_frac)
    return Workload(name=name, num_q_heads=Hq, num_kv_heads=H, head_dim=D, page_size=P, group_size=group_size,
                    sink_len=sink_len, window_len=window_len, batch=B, num_pages=num_pages,
                    max_pages_per_seq=max_pages, pages_per_split=pages_per_split,
                    seq_lens=torch.tensor(seq_lens, dtype=torch.int32), page_table=page_table, k=k, v=v,
                    tok_seq=tok_seq, tok_pos=tok_pos, slot_mapping=slot_mapping, q=q, R_k=R_k.to(device),
                    R_v=R_v.to(device), clip_k=clip_k.to(device), clip_v=clip_v.to(device), seed=seed,
                    offset_k=offset_k)


# The five workloads: sizes and distributions as their descriptions state.
CONFIG_NAMES = {
    0: "tiny_d64_L512",
    1: "b1_L32768_q32kv8_d128",
    2: "b64_Lu1024-16384_q32kv8_d128",
    3: "b4_L131072_q64kv8_d128",
    4: "append_prefill16384_decode256",
}


def config_seq_lens(cfg: int, seed: int | None = None) -> list[int]:
    seed = cfg if seed is None else seed
    if cfg == 0:
        return [512]
    if cfg == 1:
        return [32768]
    if cfg == 2:
        g = torch.Generator(device="cpu").manual_seed(seed + 77)
        return torch.randint(1024, 16385, (64,), generator=g).tolist()
    if cfg == 3:
        return [131072] * 4
    if cfg == 4:
        return [16384]
    raise ValueError(cfg)


def make_config(cfg: int, device="cpu", replicas: int = 1, seed: int | None = None) -> Workload:
    """Workload of one of the five configurations.  ``replicas`` > 1 repeats the
    batch with independent draws in disjoint pages (used to exceed the L2 cache)."""
    seed = cfg if seed is None else seed
    lens = config_seq_lens(cfg, seed) * replicas
    name = CONFIG_NAMES[cfg]
    if cfg == 0:
        return make_workload(num_q_heads=1, num_kv_heads=1, head_dim=64, group_size=32, sink_len=4,
                             window_len=32, seq_lens=lens, seed=seed, device=device, k_kind="tiny", name=name,
                             same_rotation=True)
    if cfg in (1, 2):
        return make_workload(num_q_heads=32, num_kv_heads=8, head_dim=128, group_size=64, sink_len=64,
                             window_len=128, seq_lens=lens, seed=seed, device=device, name=name)
    if cfg == 3:
        return make_workload(num_q_heads=64, num_kv_heads=8, head_dim=128, group_size=64, sink_len=64,
                             window_len=256, seq_lens=lens, seed=seed, device=device, pages_per_split=64,
                             name=name)
    if cfg == 4:
        return make_workload(num_q_heads=32, num_kv_heads=8, head_dim=128, group_size=64, sink_len=64,
                             window_len=128, seq_lens=lens, seed=seed, device=device, name=name)
    raise ValueError(cfg)


def decode_append_batch(w: Workload, n_tokens: int = 256, seed: int = 4, device=None):
    """A decode-append batch: n_tokens new K/V vectors (distributions as ``w``)
    written to distinct random slots of ``w``'s pool.  Returns (k, v, slot_mapping)."""
    device = torch.device(device) if device is not None else w.k.device
    gen_cpu = torch.Generator(device="cpu").manual_seed(seed)
    gen_dev = torch.Generator(device=device).manual_seed(seed + 1_000_003)
    H, D = w.num_kv_heads, w.head_dim
    k = _draw_k(n_tokens, H, D, gen_cpu, gen_dev, device, "qwen")
    v = _normal_bf16((n_tokens, H, D), gen_dev, device)
    slots = torch.randperm(w.num_pages * w.page_size, generator=gen_cpu)[:n_tokens].to(torch.int64)
    return k, v, slots


def calibration_samples(N: int, H: int, D: int, seed: int, kind: str = "spectrum", device="cpu") -> torch.Tensor:
    """Calibration vectors bf16 [N][H][D] for the offline calibration.
    kind 'spectrum': per head a planted covariance Q diag(lam) Q^T with Q Haar and
      lam geometric from 100 down to 0.1 (distinct, well separated eigenvalues),
      plus channel means ~N(0, 2^2): x = (z sqrt(lam)) Q^T + mu, z ~ N(0, 1);
    kind 'qwen': the K distribution of the workloads (channel means, outlier channels);
    kind 'normal': N(0, 1) (the V distribution; an isotropic covariance)."""
    gen_cpu = torch.Generator(device="cpu").manual_seed(seed)
    gen_dev = torch.Generator(device=device).manual_seed(seed + 2_000_029)
    if kind == "qwen":
        return _draw_k(N, H, D, gen_cpu, gen_dev, device, "qwen")
    if kind == "normal":
        return _normal_bf16((N, H, D), gen_dev, device)
    if kind != "spectrum":
        raise ValueError(kind)
    Q = haar_orthogonal(H, D, gen_cpu)
    lam = torch.logspace(2.0, -1.0, D, dtype=torch.float64)
    mu = 2.0 * torch.randn((H, D), dtype=torch.float64, generator=gen_cpu)
    A = (lam.sqrt().view(1, D, 1) * Q.transpose(-1, -2)).to(torch.float32).to(device)  # [H][D][D]: row j = sqrt(lam_j) q_j
    z = torch.randn((H, N, D), dtype=torch.float32, generator=gen_dev, device=device)
    x = torch.bmm(z, A) + mu.to(torch.float32).to(device).unsqueeze(1)
    return x.transpose(0, 1).contiguous().to(torch.bfloat16)


def bits16(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bf16/fp16 tensor as a numpy array (host copy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
