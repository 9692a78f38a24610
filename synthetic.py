"""Seeded synthetic inputs for the CSA layer workloads.

This module only draws random numbers and packs them into the storage formats
the layer consumes (bf16, FP8 E4M3, fp32).  It holds none of the method's
arithmetic; the oracle and the CUDA library both read the tensors it returns.

Recipe (the value distributions of the tiny decode case, reused by every
workload): compressor inputs C^a, Z^a, C^b, Z^b and the block biases B^a, B^b
are N(0,1) in bf16; the RMSNorm weight is 1 + 0.1*N(0,1); q is N(0,1); the
indexer query q^I and keys K^I are N(0,1) rounded to E4M3 (no scale); the
indexer head weights are N(0,1)/sqrt(128*64) in bf16; the sink is N(0,1) fp32.
Rows standing for an existing compressed cache or for raw window rows are
N(0,1) rows scaled to unit RMS (the distribution a RMSNorm'd latent has).
The million-token case rotates each K^I row by the orthonormal Sylvester
Hadamard matrix H_128/sqrt(128) before rounding.

Every tensor is drawn from its own torch generator, seeded by
(1000*config + sequence, tensor id), on the device the caller names, so a
sequence's inputs do not depend on the batch size.
"""
from __future__ import annotations

import dataclasses
import math

import torch

# Tensor ids: fixed per tensor so that a tensor's values do not depend on
# which other tensors are drawn.
_IDS = {name: i for i, name in enumerate([
    "Ca", "Za", "Cb", "Zb", "Ba", "Bb", "rms_w", "q", "qI", "wI", "kI", "sink", "kv", "swa",
    "Cb_prev", "Zb_prev", "ring_Ca", "ring_Za", "ring_Cb", "ring_Zb",
    "CIa", "ZIa", "CIb", "ZIb", "CIb_prev", "ZIb_prev", "BIa", "BIb", "rms_wI",
    "C", "Z", "B", "ring_CIa", "ring_ZIa", "ring_CIb", "ring_ZIb"])}

D, H, HI, DI, R = 512, 64, 64, 128, 64


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic CSA workload (shapes only)."""
    name: str
    config: int
    kind: str            # "decode" or "prefill"
    B: int
    t: int               # decode: query position; prefill: last query position
    topk: int
    n_cap: int           # compressed entries held by the cache
    Q: int = 1
    pos0: int = 0        # prefill: first query position
    m: int = 4
    W: int = 128
    hadamard_kI: bool = False


WORKLOADS = {
    0: Workload("tiny-decode-b1-1k", 0, "decode", B=1, t=1023, topk=64, n_cap=256),
    1: Workload("v4flash-decode-b32-8k", 1, "decode", B=32, t=8191, topk=512, n_cap=2048),
    2: Workload("decode-b64-128k", 2, "decode", B=64, t=131071, topk=512, n_cap=32768),
    3: Workload("v4pro-decode-b8-1m", 3, "decode", B=8, t=1048575, topk=1024, n_cap=262144,
                hadamard_kI=True),
    4: Workload("prefill-q4096-at-61440-of-64k", 4, "prefill", B=1, t=65535, topk=512, n_cap=16384,
                Q=4096, pos0=61440),
}


def _gen(seed: int, name: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1009 + _IDS[name] + 1)
    return g


def normal(shape, seed: int, name: str, device="cpu") -> torch.Tensor:
    """fp32 N(0,1) tensor from the generator of (seed, name)."""
    return torch.randn(shape, generator=_gen(seed, name, device), device=device, dtype=torch.float32)


def bf16(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16)


def e4m3(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.float8_e4m3fn)


def unit_rms_rows(x: torch.Tensor) -> torch.Tensor:
    """Scale each row (last dim) to root-mean-square 1 (input recipe only)."""
    return x * torch.rsqrt(x.pow(2).mean(-1, keepdim=True))


def hadamard(n: int, device="cpu") -> torch.Tensor:
    """Sylvester Hadamard matrix H_n (n a power of two), entries +-1."""
    h = torch.ones(1, 1, device=device)
    while h.shape[0] < n:
        h = torch.cat([torch.cat([h, h], 1), torch.cat([h, -h], 1)], 0)
    return h


def shared_params(config: int, m: int = 4, device="cpu") -> dict:
    """Layer parameters shared by all sequences: B^a, B^b, RMSNorm weight, sink."""
    s = 1000 * config
    return {
        "Ba": bf16(normal((m, D), s, "Ba", device)),
        "Bb": bf16(normal((m, D), s, "Bb", device)),
        "rms_w": bf16(1.0 + 0.1 * normal((D,), s, "rms_w", device)),
        "sink": normal((H,), s, "sink", device),
    }


def _per_seq(B, config, name, shape, device, make):
    return torch.stack([make(normal(shape, 1000 * config + b, name, device)) for b in range(B)])


def compressor_rows(config: int, B: int, T: int, device="cpu", names=("Ca", "Za", "Cb", "Zb")) -> dict:
    """[B, T, D] bf16 N(0,1) compressor inputs for T consecutive tokens."""
    return {n: _per_seq(B, config, n, (T, D), device, bf16) for n in names}


def indexer_compressor_inputs(config: int, B: int, T: int, m: int = 4, device="cpu") -> dict:
    """The indexer key compressor's inputs (width 128): rows CIa, ZIa, CIb,
    ZIb [B, T, 128] and the m rows before the chunk, N(0,1) bf16; block biases
    BIa, BIb [m, 128] N(0,1) bf16; RMSNorm weight 1 + 0.1*N(0,1)."""
    s = 1000 * config
    out = {n: _per_seq(B, config, n, (T, DI), device, bf16) for n in ("CIa", "ZIa", "CIb", "ZIb")}
    out.update({n: _per_seq(B, config, n, (m, DI), device, bf16) for n in ("CIb_prev", "ZIb_prev")})
    out["BIa"] = bf16(normal((m, DI), s, "BIa", device))
    out["BIb"] = bf16(normal((m, DI), s, "BIb", device))
    out["rms_wI"] = bf16(1.0 + 0.1 * normal((DI,), s, "rms_wI", device))
    return out


def indexer_ring_inputs(config: int, B: int, m: int = 4, device="cpu") -> dict:
    """The indexer key compressor's decode staging ring: ring_CIa, ring_ZIa,
    ring_CIb, ring_ZIb [B, 2m, 128] N(0,1) bf16 (slot u mod 2m holds token
    u's row), with the block biases and RMSNorm weight of
    indexer_compressor_inputs."""
    s = 1000 * config
    out = {n: _per_seq(B, config, n, (2 * m, DI), device, bf16) for n in ("ring_CIa", "ring_ZIa", "ring_CIb",
                                                                          "ring_ZIb")}
    out["BIa"] = bf16(normal((m, DI), s, "BIa", device))
    out["BIb"] = bf16(normal((m, DI), s, "BIb", device))
    out["rms_wI"] = bf16(1.0 + 0.1 * normal((DI,), s, "rms_wI", device))
    return out


def indexer_query(config: int, B: int, Q: int, device="cpu") -> dict:
    return {
        "qI": _per_seq(B, config, "qI", (Q, HI, DI), device, e4m3),
        "wI": _per_seq(B, config, "wI", (Q, HI), device, lambda x: bf16(x / math.sqrt(DI * HI))),
    }


def indexer_keys(config: int, B: int, n: int, device="cpu", hadamard_rows: bool = False) -> torch.Tensor:
    if hadamard_rows:
        Hm = hadamard(DI, device) / math.sqrt(DI)
        return _per_seq(B, config, "kI", (n, DI), device, lambda x: e4m3(x @ Hm.T))
    return _per_seq(B, config, "kI", (n, DI), device, e4m3)


def indexer_query_bf16(config: int, B: int, Q: int, device="cpu") -> dict:
    """indexer_query's draws as bf16 rows (the FP4 indexer quantizes them)."""
    return {
        "qI": _per_seq(B, config, "qI", (Q, HI, DI), device, bf16),
        "wI": _per_seq(B, config, "wI", (Q, HI), device, lambda x: bf16(x / math.sqrt(DI * HI))),
    }


def indexer_keys_bf16(config: int, B: int, n: int, device="cpu") -> torch.Tensor:
    """indexer_keys' draws as bf16 rows (the FP4 indexer quantizes them)."""
    return _per_seq(B, config, "kI", (n, DI), device, bf16)


def main_query(config: int, B: int, Q: int, device="cpu") -> torch.Tensor:
    return _per_seq(B, config, "q", (Q, H, D), device, bf16)


def cache_rows(config: int, B: int, n: int, device="cpu", name="kv") -> torch.Tensor:
    """Existing compressed cache / raw window rows: unit-RMS N(0,1) rows, bf16."""
    return _per_seq(B, config, name, (n, D), device, lambda x: bf16(unit_rms_rows(x)))


def single_stream_inputs(config: int, B: int, T: int, m: int, bias: bool = True, device="cpu") -> dict:
    """The single-stream (HCA / CSA2) compressor's inputs: rows C, Z [B, T,
    512] N(0,1) bf16; slot bias B [m, 512] N(0,1) bf16 (None without bias);
    RMSNorm weight 1 + 0.1*N(0,1)."""
    s = 1000 * config
    return {"C": _per_seq(B, config, "C", (T, D), device, bf16), "Z": _per_seq(B, config, "Z", (T, D), device, bf16),
            "B": bf16(normal((m, D), s, "B", device)) if bias else None,
            "rms_w": bf16(1.0 + 0.1 * normal((D,), s, "rms_w", device))}


def decode_inputs(w: Workload, device="cpu", B: int | None = None) -> dict:
    """Inputs of one decode step (the query at position w.t for each sequence).

    The cache holds entries 0..n_cap-1 as unit-RMS rows (the entry the step
    emits, V(t)-1 when (t+1) % m == 0, is overwritten by the step), the indexer
    keys for all n_cap entries, the staging rings of the last 2m tokens'
    compressor rows (main and indexer-key compressors), the window ring and
    the queries.
    """
    B = w.B if B is None else B
    c = w.config
    out = shared_params(c, w.m, device)
    out.update(indexer_query(c, B, 1, device))
    out["kI"] = indexer_keys(c, B, w.n_cap, device, w.hadamard_kI)
    out["kv"] = cache_rows(c, B, w.n_cap, device)
    out["swa"] = cache_rows(c, B, w.W, device, name="swa")
    out["q"] = main_query(c, B, 1, device)
    out.update({k: v for k, v in zip(
        ("ring_Ca", "ring_Za", "ring_Cb", "ring_Zb"),
        compressor_rows(c, B, 2 * w.m, device, names=("ring_Ca", "ring_Za", "ring_Cb", "ring_Zb")).values())})
    out.update(indexer_ring_inputs(c, B, w.m, device))
    out["q_pos"] = torch.full((B, 1), w.t, dtype=torch.int32, device=device)
    return out


def prefill_inputs(w: Workload, device="cpu", Q: int | None = None) -> dict:
    """Inputs of one prefill chunk of Q tokens at positions pos0.. (B sequences).

    The cache holds pos0/m existing entries (unit-RMS rows); the chunk's
    compressor rows produce the next Q/m entries.  Indexer keys are given for
    every entry up to (pos0+Q)/m, and the indexer key compressor's rows of the
    chunk (CIa..ZIb, CIb_prev, ZIb_prev) for the calls that compute the
    chunk's keys.  The window buffer is linear: row j is position
    pos0-(W-1)+j.
    """
    Q = w.Q if Q is None else Q
    c, B, m = w.config, w.B, w.m
    n_cap = (w.pos0 + Q) // m
    out = shared_params(c, m, device)
    out.update(compressor_rows(c, B, Q, device))
    prev = compressor_rows(c, B, m, device, names=("Cb_prev", "Zb_prev"))
    out["Cb_prev"], out["Zb_prev"] = prev["Cb_prev"], prev["Zb_prev"]
    out.update(indexer_query(c, B, Q, device))
    out["kI"] = indexer_keys(c, B, n_cap, device, w.hadamard_kI)
    out["kv"] = cache_rows(c, B, n_cap, device)
    out["swa"] = cache_rows(c, B, w.W - 1 + Q, device, name="swa")
    out["q"] = main_query(c, B, Q, device)
    out.update(indexer_compressor_inputs(c, B, Q, m, device))
    out["n_cap"] = n_cap
    return out


def bits(t: torch.Tensor):
    """Raw storage bits of a tensor as a numpy array (uint16 for bf16, uint8 for
    e4m3, unchanged otherwise) — the form the oracle reads."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.numpy()
