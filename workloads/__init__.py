"""Seeded synthetic inputs for the shared-input batched linear.

This module is shared by the tests, the benchmark and the smoke check, on both
sides of a parity comparison.  It holds no arithmetic of the method itself (no
dequantisation, no dot product): only random draws, the quantiser that turns
an fp32 draw into Q8/Q4 storage, and the host byte encodings that
``il_upload_weight`` and the oracle both read.

Recipe (the same for every workload):
  * ``g = torch.Generator().manual_seed(seed)`` on the CPU, seed 0 by default;
  * ``x = randn(t, n_in)`` fp32 from ``g`` first, then for each job in order
    ``W_j = 0.02 * randn(n_out_j, n_in)`` fp32 from the same ``g``;
  * bf16 storage is ``W_j`` rounded to nearest-even bf16;
  * Q8 / Q4 storage quantises the fp32 draw per (row, 32-block):
    ``amax = max |w|``, ``d = amax / 127`` (Q8) or ``amax / 7`` (Q4), and
    ``q = clamp(round_half_even(w / d), -127..127 | -7..7)``; ``amax == 0``
    gives ``d = 0, q = 0``.

Host byte layouts (one contiguous buffer per weight, ``[n_out, n_in]``):
  * bf16: ``u16 w[n_out][n_in]``
  * Q8:   ``i8 q[n_out][n_in]`` then ``f32 d[n_out][n_in/32]``
  * Q4:   ``u8 p[n_out][n_in/2]`` (element 2k in bits 0-3 of byte k, element
    2k+1 in bits 4-7, two's complement) then ``f32 d[n_out][n_in/32]``
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

W_STD = 0.02
BLOCK = 32


# ---------------------------------------------------------------------------
# workload table: the shapes of the decoder batches this library serves
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class Batch:
    """One ``il_matmul_batch`` call: jobs over one shared x."""
    name: str
    n_in: int
    n_outs: tuple


@dataclass(frozen=True)
class Workload:
    name: str
    fmts: tuple
    ts: tuple
    batches: tuple
    note: str = ""
    fused: bool = False   # each batch's two jobs run as one fused gate+up job (h = gelu(g) * u)


TINY = Workload("tiny_bf16", ("bf16",), (1, 4),
                (Batch("tiny", 256, (512, 256)),),
                "two jobs over n_in=256; L2-resident")
DECODE_BF16 = Workload("decode_bf16_qkv_gateup", ("bf16",), (1,),
                       (Batch("qkv", 4096, (4096, 1024, 1024)),
                        Batch("gate_up", 4096, (12288, 12288))),
                       "single-token decode, attention projections then gate+up")
DECODE_QUANT = Workload("decode_quant_qkv_gateup_down", ("q8", "q4"), (1, 8),
                        (Batch("qkv", 4096, (4096, 1024, 1024)),
                         Batch("gate_up", 4096, (12288, 12288)),
                         Batch("down", 12288, (4096,))),
                        "quantised decode, t=1 and t=8")
PREFILL_BF16 = Workload("prefill_bf16_gateup_down", ("bf16",), (512, 2048),
                        (Batch("gate_up", 4096, (12288, 12288)),
                         Batch("down", 12288, (4096,))),
                        "prompt prefill, tensor-core regime")
PREFILL_QUANT = Workload("prefill_quant_gateup_down", ("q8", "q4"), (512,),
                         (Batch("gate_up", 4096, (12288, 12288)),
                          Batch("down", 12288, (4096,))),
                         "prompt prefill with quantised weights")
VOCAB = Workload("vocab_projection", ("bf16", "q4"), (1, 8),
                 (Batch("vocab", 2560, (262144,)),),
                 "one very tall job")

GATE_UP_FUSED = Workload("gate_up_fused", ("bf16", "q8", "q4"), (1, 8, 512),
                         (Batch("gate_up", 4096, (12288, 12288)),),
                         "gate+up as one fused job writing h = gelu(g) * u", fused=True)

WORKLOADS = (TINY, DECODE_BF16, DECODE_QUANT, PREFILL_BF16, VOCAB, PREFILL_QUANT, GATE_UP_FUSED)
BY_NAME = {w.name: w for w in WORKLOADS}


@dataclass(frozen=True)
class HeadConfig:
    """A centroid-masked LM head: the vocabulary in n_cent clusters of vocab / n_cent tokens."""
    name: str
    h: int
    vocab: int
    n_cent: int
    top_k: int
    note: str = ""


# the dense vocab projection's shape (2560 -> 262144), in 4096 clusters of 64 tokens
CENTROID_HEAD = HeadConfig("centroid_lm_head", 2560, 262144, 4096, 32,
                           "top 32 of 4096 clusters scored: 2048 of 262144 vocabulary rows")


# ---------------------------------------------------------------------------
# encodings
# ---------------------------------------------------------------------------
def weight_bytes(fmt: str, n_out: int, n_in: int) -> int:
    if fmt == "bf16":
        return 2 * n_out * n_in
    if fmt == "q8":
        return n_out * n_in + 4 * n_out * (n_in // BLOCK)
    if fmt == "q4":
        return n_out * (n_in // 2) + 4 * n_out * (n_in // BLOCK)
    raise ValueError(fmt)


def bf16_bits(w: torch.Tensor) -> np.ndarray:
    """fp32 tensor -> u16 bit patterns of its nearest-even bf16 rounding."""
    return w.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def encode_bf16(bits: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(bits, dtype=np.uint16).reshape(-1).view(np.uint8)


def encode_q8(q: np.ndarray, d: np.ndarray) -> np.ndarray:
    """``q`` int8-valued ``[n_out][n_in]``, ``d`` fp32 ``[n_out][n_in/32]`` -> host bytes."""
    q = np.ascontiguousarray(q).astype(np.int8)
    d = np.ascontiguousarray(d, dtype=np.float32)
    n_out, n_in = q.shape
    assert n_in % BLOCK == 0 and d.shape == (n_out, n_in // BLOCK)
    return np.concatenate([q.reshape(-1).view(np.uint8), d.reshape(-1).view(np.uint8)])


def pack_nibbles(q: np.ndarray) -> np.ndarray:
    """Signed 4-bit values ``[n_out][n_in]`` -> bytes ``[n_out][n_in/2]``, low nibble first."""
    q = np.asarray(q)
    nib = (q.astype(np.int16) & 0xF).astype(np.uint8)
    return (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)


def encode_q4(q: np.ndarray, d: np.ndarray) -> np.ndarray:
    """``q`` in [-8, 7] ``[n_out][n_in]``, ``d`` fp32 ``[n_out][n_in/32]`` -> host bytes."""
    q = np.asarray(q)
    n_out, n_in = q.shape
    assert n_in % BLOCK == 0 and d.shape == (n_out, n_in // BLOCK)
    assert q.min(initial=0) >= -8 and q.max(initial=0) <= 7
    p = pack_nibbles(q)
    d = np.ascontiguousarray(d, dtype=np.float32)
    return np.concatenate([p.reshape(-1), d.reshape(-1).view(np.uint8)])


def quantize(w: torch.Tensor, qmax: int):
    """Symmetric per-(row, 32-block) quantiser on an fp32 ``[n_out][n_in]`` tensor."""
    n_out, n_in = w.shape
    wb = w.reshape(n_out, n_in // BLOCK, BLOCK)
    amax = wb.abs().amax(dim=2)
    d = amax / float(qmax)
    safe = torch.where(d > 0, d, torch.ones_like(d))
    q = torch.round(wb / safe.unsqueeze(2)).clamp_(-qmax, qmax)
    q = torch.where((d > 0).unsqueeze(2), q, torch.zeros_like(q))
    return q.reshape(n_out, n_in).to(torch.int8).numpy(), d.numpy().astype(np.float32)


def encode_weight(fmt: str, w: torch.Tensor) -> np.ndarray:
    """fp32 draw -> host bytes in ``fmt``."""
    if fmt == "bf16":
        return encode_bf16(bf16_bits(w))
    if fmt == "q8":
        q, d = quantize(w, 127)
        return encode_q8(q, d)
    if fmt == "q4":
        q, d = quantize(w, 7)
        return encode_q4(q, d)
    raise ValueError(fmt)


# ---------------------------------------------------------------------------
# seeded draws
# ---------------------------------------------------------------------------
@dataclass
class BatchInputs:
    fmt: str
    t: int
    n_in: int
    x: np.ndarray                      # fp32 [t][n_in]
    jobs: list = field(default_factory=list)   # [(fmt, host_bytes u8, n_out)]
    fused: bool = False                # jobs are (gate, up) of one fused gate+up job

    @property
    def weight_bytes(self) -> int:
        return sum(int(w.size) for _, w, _ in self.jobs)

    @property
    def flops(self) -> int:
        return 2 * self.t * self.n_in * sum(n for _, _, n in self.jobs)


def make_batch(n_in: int, n_outs, t: int, fmt: str, seed: int = 0,
               x_scale: float = 1.0) -> BatchInputs:
    """Draw x and every W_j of one batch from a fresh generator seeded ``seed``."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(t, n_in, generator=g, dtype=torch.float32) * x_scale
    out = BatchInputs(fmt, t, n_in, x.numpy().copy())
    for n_out in n_outs:
        w = torch.randn(n_out, n_in, generator=g, dtype=torch.float32) * W_STD
        out.jobs.append((fmt, encode_weight(fmt, w), n_out))
    return out


def make_workload_batch(workload: Workload, batch: Batch, t: int, fmt: str,
                        seed: int = 0) -> BatchInputs:
    assert fmt in workload.fmts and t in workload.ts
    b = make_batch(batch.n_in, batch.n_outs, t, fmt, seed)
    b.fused = workload.fused
    return b


def make_x(t: int, n_in: int, seed: int) -> np.ndarray:
    g = torch.Generator().manual_seed(seed)
    return torch.randn(t, n_in, generator=g, dtype=torch.float32).numpy().copy()


@dataclass
class HeadInputs:
    h: int
    vocab: int
    n_cent: int
    x: np.ndarray            # fp32 [h]
    centroids: np.ndarray    # bf16 host bytes [n_cent][h]
    embed: np.ndarray        # bf16 host bytes [vocab][h]
    ordering: np.ndarray     # u32 [vocab], a permutation: cluster c owns [c*per, (c+1)*per)


def make_head_inputs(h: int, vocab: int, n_cent: int, seed: int = 0) -> HeadInputs:
    """x = randn(h), centroids = 0.02*randn(n_cent, h), embed = 0.02*randn(vocab, h) (both
    rounded to bf16), ordering = a random permutation, all from one seeded generator."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(h, generator=g, dtype=torch.float32)
    cen = torch.randn(n_cent, h, generator=g, dtype=torch.float32) * W_STD
    emb = torch.randn(vocab, h, generator=g, dtype=torch.float32) * W_STD
    order = torch.randperm(vocab, generator=g).numpy().astype(np.uint32)
    return HeadInputs(h, vocab, n_cent, x.numpy().copy(), encode_bf16(bf16_bits(cen)),
                      encode_bf16(bf16_bits(emb)), order)
