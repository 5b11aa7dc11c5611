"""Seeded synthetic workloads for the DSA verify / draft step.

This module only draws random inputs (shapes, lengths, values); it holds none
of the method's arithmetic.  The tests and the benchmark feed the same arrays
to the CUDA path and to the CPU oracle.  Each tensor has its own random stream
derived from (seed, tensor name), drawn with torch's CPU generator seeded per
stream, so any tensor can be regenerated on its own.

Workloads (shapes of the MTP decode step of a GLM-5.x / DeepSeek-V3.2 style
model: index_topk 2048, 576-wide latent = 512 + 64, 64 indexer heads of 128,
128 query heads, 1 bonus + 5 draft tokens per request):

* ``tiny``   2 requests, contexts 100 and 300, 3 drafts (4 verify rows each),
             8 query heads, float32 latent, float32 indexer 4 x 64, top-k 32.
* ``verify`` 32 requests x 8192 cached tokens, 6 verify rows each, bf16 latent,
             FP8 indexer 64 x 128 with block-128 scales, top-k 2048.
* ``draft``  64 requests x 32768, four 1-row draft forwards with the step-0
             top-k shared by steps 1-3, accepted-segment write-back first.
* ``long``   8 requests, contexts log-uniform in [4096, 1048576], 6 rows each.
* ``decode`` 128 requests, contexts log-uniform in [1024, 131072]: merge,
             6-row verify, greedy acceptance (mean accept length about 2.76),
             write-back and four shared-index draft steps.

Value recipe: activations ~ N(0, 1) (``tiny``: N(0, 1)/sqrt(d)); head weights
~ U(0, 1); token ids uniform over the vocabulary; target argmax equals the
draft token at each position independently with probability p (0.7 for
``tiny``, 0.67065 elsewhere, which gives 1 + sum_{i=1..5} p^i = 2.76), else a
different token; the argmax after the last draft (the bonus) is uniform.
"""
from __future__ import annotations

import dataclasses
import math
import zlib
from typing import Dict, List, Optional

import numpy as np
import torch

SOFTMAX_SCALE = 1.0 / math.sqrt(576.0)
ACCEPT_P = 0.67065
GLM_VOCAB = 154880


@dataclasses.dataclass
class Spec:
    name: str
    seed: int
    B: int
    lengths: Optional[List[int]]       # fixed lengths, or None for log-uniform
    len_range: Optional[tuple]         # (lo, hi) for log-uniform lengths
    K: int                             # draft tokens per request (verify rows = K + 1)
    H_Q: int
    latent_f32: bool                   # float32 latent and float32 indexer (no FP8)
    H_I: int
    D_I: int
    topk: int
    vocab: int
    accept_p: float
    draft_steps: int = 0               # shared-index draft forwards after acceptance
    verify: bool = True                # has a multi-row verify step
    scaled_normal: bool = False        # N(0,1)/sqrt(d) instead of N(0,1)


SPECS: Dict[str, Spec] = {
    "tiny": Spec("tiny", 0, 2, [100, 300], None, 3, 8, True, 4, 64, 32, 1000, 0.7,
                 draft_steps=4, scaled_normal=True),
    "verify": Spec("verify", 1, 32, [8192] * 32, None, 5, 128, False, 64, 128, 2048,
                   GLM_VOCAB, ACCEPT_P, draft_steps=4),
    "draft": Spec("draft", 2, 64, [32768] * 64, None, 5, 128, False, 64, 128, 2048,
                  GLM_VOCAB, ACCEPT_P, draft_steps=4, verify=False),
    "long": Spec("long", 3, 8, None, (4096, 1048576), 5, 128, False, 64, 128, 2048,
                 GLM_VOCAB, ACCEPT_P),
    "decode": Spec("decode", 4, 128, None, (1024, 131072), 5, 128, False, 64, 128, 2048,
                   GLM_VOCAB, ACCEPT_P, draft_steps=4),
}


def _stream(seed: int, name: str) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed((seed * 1_000_003 + zlib.crc32(name.encode())) % (2 ** 63))
    return g


def normal(seed: int, name: str, shape, std: float = 1.0, dtype=torch.float32) -> torch.Tensor:
    """N(0, std^2) samples, generated in float32 then cast to dtype (CPU)."""
    g = _stream(seed, name)
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def uniform(seed: int, name: str, shape, lo=0.0, hi=1.0) -> torch.Tensor:
    g = _stream(seed, name)
    return torch.rand(*shape, generator=g, dtype=torch.float32) * (hi - lo) + lo


def integers(seed: int, name: str, shape, lo: int, hi: int) -> torch.Tensor:
    g = _stream(seed, name)
    return torch.randint(lo, hi, tuple(shape), generator=g, dtype=torch.int64)


@dataclasses.dataclass
class Workload:
    spec: Spec
    L: np.ndarray              # [B] committed context before the step
    r: int                     # verify rows per request (K + 1)
    cap: np.ndarray            # [B] cache tokens reserved per request
    cache_start: np.ndarray    # [B] int64 pool offset
    T: int                     # pool tokens
    # verify rows
    row_req: np.ndarray        # [R] int32
    row_pos: np.ndarray        # [R] int64
    # tokens
    prompt_tokens: np.ndarray  # [B] int64 (1 input token per request)
    prompt_offsets: np.ndarray  # [B+1] uint32
    draft_tokens: np.ndarray   # [B, K] int64
    target_argmax: np.ndarray  # [B, K+1] int64
    # raw activations (CPU torch tensors)
    tensors: Dict[str, torch.Tensor]

    @property
    def B(self):
        return self.spec.B

    @property
    def R(self):
        return len(self.row_req)


def lengths_for(spec: Spec) -> np.ndarray:
    if spec.lengths is not None:
        return np.asarray(spec.lengths, dtype=np.int64)
    lo, hi = spec.len_range
    u = uniform(spec.seed, "lengths", (spec.B,)).double().numpy()
    return np.floor(np.exp(np.log(lo) + u * (np.log(hi) - np.log(lo)))).astype(np.int64)


def synthetic_argmax(seed: int, draft: torch.Tensor, vocab: int, p: float) -> torch.Tensor:
    """Target argmax [B, K+1]: matches draft[b, i] with probability p, else a
    different token; the last column is uniform."""
    B, K = draft.shape
    match = uniform(seed, "argmax_match", (B, K)) < p
    other = (draft + 1 + integers(seed, "argmax_other", (B, K), 0, vocab - 1)) % vocab
    head = torch.where(match, draft, other)
    bonus = integers(seed, "argmax_bonus", (B, 1), 0, vocab)
    return torch.cat([head, bonus], dim=1)


def build(name_or_spec, with_tensors: bool = True) -> Workload:
    spec = SPECS[name_or_spec] if isinstance(name_or_spec, str) else name_or_spec
    s = spec.seed
    B, K = spec.B, spec.K
    L = lengths_for(spec)
    r = K + 1 if spec.verify else 1
    extra = (K + 1) + spec.draft_steps + 1      # verify window + draft appends
    cap = L + extra
    cache_start = np.zeros(B, dtype=np.int64)
    cache_start[1:] = np.cumsum(cap)[:-1]
    T = int(cap.sum())
    row_req = np.repeat(np.arange(B, dtype=np.int32), r)
    row_pos = (np.repeat(L, r) + np.tile(np.arange(r), B)).astype(np.int64)

    prompt = integers(s, "prompt_tokens", (B,), 0, spec.vocab)
    offsets = np.arange(B + 1, dtype=np.uint32)
    draft = integers(s, "draft_tokens", (B, K), 0, spec.vocab)
    argmax = synthetic_argmax(s, draft, spec.vocab, spec.accept_p)

    std_i = 1.0 / math.sqrt(spec.D_I) if spec.scaled_normal else 1.0
    std_l = 1.0 / math.sqrt(576.0) if spec.scaled_normal else 1.0
    lat_dtype = torch.float32 if spec.latent_f32 else torch.bfloat16
    R = len(row_req)
    tensors: Dict[str, torch.Tensor] = {}
    if with_tensors:
        tensors["q_idx"] = normal(s, "q_idx", (R, spec.H_I, spec.D_I), std_i)
        tensors["w_idx"] = uniform(s, "w_idx", (R, spec.H_I))
        tensors["k_idx"] = normal(s, "k_idx", (T, spec.D_I), std_i)
        tensors["latent"] = normal(s, "latent", (T, 576), std_l, lat_dtype)
        tensors["q_mla"] = normal(s, "q_mla", (R, spec.H_Q, 576), std_l, lat_dtype)
    return Workload(spec, L, r, cap, cache_start, T, row_req, row_pos,
                    prompt.numpy(), offsets, draft.numpy(), argmax.numpy(), tensors)


def draft_tensors(w: Workload, with_pool: bool = True) -> Dict[str, torch.Tensor]:
    """Inputs of the draft layer for the accepted-segment write-back and the
    shared-index draft loop: a separate draft pool (latent + indexer key), the
    6-row window of draft-layer KV to write back, and per-step queries."""
    spec = w.spec
    s = spec.seed
    B, W = spec.B, spec.K + 1
    std_i = 1.0 / math.sqrt(spec.D_I) if spec.scaled_normal else 1.0
    std_l = 1.0 / math.sqrt(576.0) if spec.scaled_normal else 1.0
    lat_dtype = torch.float32 if spec.latent_f32 else torch.bfloat16
    t: Dict[str, torch.Tensor] = {}
    if with_pool:
        t["d_k_idx"] = normal(s, "d_k_idx", (w.T, spec.D_I), std_i)
        t["d_latent"] = normal(s, "d_latent", (w.T, 576), std_l, lat_dtype)
    t["src_latent"] = normal(s, "src_latent", (B, W, 576), std_l, lat_dtype)
    t["src_k_idx"] = normal(s, "src_k_idx", (B, W, spec.D_I), std_i)
    t["d_q_idx"] = normal(s, "d_q_idx", (B, spec.H_I, spec.D_I), std_i)
    t["d_w_idx"] = uniform(s, "d_w_idx", (B, spec.H_I))
    for j in range(spec.draft_steps):
        t[f"d_q_mla{j}"] = normal(s, f"d_q_mla{j}", (B, spec.H_Q, 576), std_l, lat_dtype)
    return t
