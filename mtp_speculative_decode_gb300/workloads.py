"""Seeded synthetic workloads for the DSA verify / draft step.

This module only draws random inputs (shapes, lengths, values); it holds none
of the method's arithmetic.  The tests and the benchmark feed the same arrays
to the CUDA path and to the CPU oracle.  Each tensor has its own random stream
derived from (seed, tensor name), drawn with torch's CPU generator seeded per
stream, so any tensor can be regenerated on its own.

Generation: every tensor is drawn in blocks of 65536 consecutive elements
(row-major), block i from its own numpy PCG64 stream seeded by (workload seed,
CRC-32 of the tensor name, i).  Any range of rows can therefore be regenerated
on its own (the oracle reads only the requests it checks), the blocks are
drawn in parallel threads, and a device copy is filled chunk by chunk without
a full host copy.  Normal values are float32 samples (then rounded to the
tensor's dtype, bf16 by round-to-nearest-even); uniforms are float32.

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
import os
import threading
import zlib
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, List, Optional

import numpy as np
import torch

SOFTMAX_SCALE = 1.0 / math.sqrt(576.0)
ACCEPT_P = 0.67065
GLM_VOCAB = 154880
BLOCK = 1 << 16                     # elements per random stream


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


# ----------------------------------------------------------------------------- block streams

def _key(name: str) -> int:
    return zlib.crc32(name.encode())


def _block_rng(seed: int, name: str, block: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, _key(name), block])))


def _draw(seed: int, name: str, kind: str, e0: int, e1: int) -> np.ndarray:
    """Elements [e0, e1) of a tensor's float32 stream ("normal" or "uniform")."""
    out = np.empty(e1 - e0, dtype=np.float32)
    b = e0 // BLOCK
    pos = 0
    while pos < e1 - e0:
        lo = b * BLOCK
        g = _block_rng(seed, name, b)
        blk = g.standard_normal(BLOCK, dtype=np.float32) if kind == "normal" else g.random(BLOCK, dtype=np.float32)
        a = max(e0, lo) - lo
        n = min(e1, lo + BLOCK) - lo - a
        out[pos:pos + n] = blk[a:a + n]
        pos += n
        b += 1
    return out


_POOL = None
_POOL_LOCK = threading.Lock()


def _pool() -> ThreadPoolExecutor:
    global _POOL
    with _POOL_LOCK:
        if _POOL is None:
            _POOL = ThreadPoolExecutor(max(1, min(32, os.cpu_count() or 1)))
        return _POOL


def normal(seed: int, name: str, shape, std: float = 1.0, dtype=torch.float32) -> torch.Tensor:
    """N(0, std^2) samples of the given shape (CPU), from the tensor's block streams."""
    return TensorSpec(tuple(shape), "normal", std, dtype).generate(seed, name)


def uniform(seed: int, name: str, shape, lo=0.0, hi=1.0) -> torch.Tensor:
    x = TensorSpec(tuple(shape), "uniform", 1.0, torch.float32).generate(seed, name)
    return x * (hi - lo) + lo


def integers(seed: int, name: str, shape, lo: int, hi: int) -> torch.Tensor:
    """Uniform integers in [lo, hi) (one stream per tensor: these tensors are small)."""
    g = _block_rng(seed, name, 0)
    return torch.from_numpy(g.integers(lo, hi, tuple(shape), dtype=np.int64))


@dataclasses.dataclass
class TensorSpec:
    shape: tuple
    kind: str            # "normal" or "uniform"
    std: float
    dtype: torch.dtype

    @property
    def row_elems(self) -> int:
        return int(np.prod(self.shape[1:], dtype=np.int64)) if len(self.shape) > 1 else 1

    def _rows_f32(self, seed, name, a, b) -> np.ndarray:
        x = _draw(seed, name, self.kind, a * self.row_elems, b * self.row_elems)
        if self.std != 1.0:
            x *= np.float32(self.std)
        return x

    def _cast(self, x: np.ndarray, rows: int) -> torch.Tensor:
        t = torch.from_numpy(x).reshape((rows,) + tuple(self.shape[1:]))
        return t if self.dtype == torch.float32 else t.to(self.dtype)

    def rows(self, seed, name, a: int, b: int) -> torch.Tensor:
        """Rows [a, b) along the first dimension, generated in parallel blocks."""
        a, b = max(0, a), min(self.shape[0], b)
        if b <= a:
            return self._cast(np.empty(0, np.float32), 0)
        per = max(1, (1 << 22) // self.row_elems)          # about 4M elements per task
        starts = list(range(a, b, per))
        parts = list(_pool().map(lambda s: self._cast(self._rows_f32(seed, name, s, min(b, s + per)),
                                                      min(b, s + per) - s), starts))
        return parts[0] if len(parts) == 1 else torch.cat(parts)

    def generate(self, seed, name) -> torch.Tensor:
        return self.rows(seed, name, 0, self.shape[0]) if len(self.shape) else \
            self._cast(self._rows_f32(seed, name, 0, 1), 1).reshape(())

    def to_device(self, seed, name, device) -> torch.Tensor:
        """The tensor on `device`, filled in chunks (about 64M elements each) as they are generated."""
        out = torch.empty(self.shape, dtype=self.dtype, device=device)
        n = self.shape[0]
        per = max(1, (1 << 26) // self.row_elems)
        for s in range(0, n, per):
            e = min(n, s + per)
            out[s:e].copy_(self.rows(seed, name, s, e))
        return out


class Tensors:
    """The named input tensors of a workload, generated on demand.

    t[name] is the whole tensor (CPU, cached); t.rows(name, a, b) and
    t.take(name, index) regenerate only the rows asked for;
    t.to_device(name, device) fills a device tensor chunk by chunk."""

    def __init__(self, seed: int, specs: Dict[str, TensorSpec]):
        self.seed = seed
        self.specs = specs
        self._cache: Dict[str, torch.Tensor] = {}

    def __contains__(self, name):
        return name in self.specs

    def __iter__(self):
        return iter(self.specs)

    def keys(self):
        return self.specs.keys()

    def __getitem__(self, name) -> torch.Tensor:
        if name not in self._cache:
            self._cache[name] = self.specs[name].generate(self.seed, name)
        return self._cache[name]

    def shape(self, name):
        return self.specs[name].shape

    def rows(self, name, a: int, b: int) -> torch.Tensor:
        if name in self._cache:
            return self._cache[name][a:b]
        return self.specs[name].rows(self.seed, name, a, b)

    def take(self, name, index) -> torch.Tensor:
        """Rows at the given first-dimension indices (in that order)."""
        idx = np.asarray(index, dtype=np.int64).reshape(-1)
        if name in self._cache:
            return self._cache[name][torch.from_numpy(idx)]
        if len(idx) == 0:
            return self.rows(name, 0, 0)
        # regenerate the covering block ranges once, then gather
        spec = self.specs[name]
        per = max(1, BLOCK // spec.row_elems)
        uniq = np.unique(idx // per)
        spans = []
        for u in uniq:
            if spans and spans[-1][1] == u:
                spans[-1][1] = u + 1
            else:
                spans.append([u, u + 1])
        parts, rowmap, base = [], {}, 0
        for u0, u1 in spans:
            a, b = int(u0 * per), int(min(spec.shape[0], u1 * per))
            parts.append(self.rows(name, a, b))
            rowmap[(a, b)] = base
            base += b - a
        cat = torch.cat(parts) if len(parts) > 1 else parts[0]
        pos = np.empty_like(idx)
        starts = np.array([k[0] for k in rowmap], dtype=np.int64)
        offs = np.array(list(rowmap.values()), dtype=np.int64)
        j = np.searchsorted(starts, idx, side="right") - 1
        pos[:] = offs[j] + (idx - starts[j])
        return cat[torch.from_numpy(pos)]

    def to_device(self, name, device) -> torch.Tensor:
        if name in self._cache:
            return self._cache[name].to(device).contiguous()
        return self.specs[name].to_device(self.seed, name, device)


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
    # activations and caches (generated on demand, see Tensors)
    tensors: Tensors

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


def _tensor_specs(spec: Spec, R: int, T: int) -> Dict[str, TensorSpec]:
    std_i = 1.0 / math.sqrt(spec.D_I) if spec.scaled_normal else 1.0
    std_l = 1.0 / math.sqrt(576.0) if spec.scaled_normal else 1.0
    lat = torch.float32 if spec.latent_f32 else torch.bfloat16
    f32 = torch.float32
    t = {
        "q_idx": TensorSpec((R, spec.H_I, spec.D_I), "normal", std_i, f32),
        "w_idx": TensorSpec((R, spec.H_I), "uniform", 1.0, f32),
        "k_idx": TensorSpec((T, spec.D_I), "normal", std_i, f32),
        "latent": TensorSpec((T, 576), "normal", std_l, lat),
        "q_mla": TensorSpec((R, spec.H_Q, 576), "normal", std_l, lat),
    }
    if spec.draft_steps:
        B, W = spec.B, spec.K + 1
        t.update({
            "d_k_idx": TensorSpec((T, spec.D_I), "normal", std_i, f32),
            "d_latent": TensorSpec((T, 576), "normal", std_l, lat),
            "src_latent": TensorSpec((B, W, 576), "normal", std_l, lat),
            "src_k_idx": TensorSpec((B, W, spec.D_I), "normal", std_i, f32),
            "d_q_idx": TensorSpec((B, spec.H_I, spec.D_I), "normal", std_i, f32),
            "d_w_idx": TensorSpec((B, spec.H_I), "uniform", 1.0, f32),
        })
        for j in range(spec.draft_steps):
            t[f"d_q_mla{j}"] = TensorSpec((B, spec.H_Q, 576), "normal", std_l, lat)
    return t


def build(name_or_spec) -> Workload:
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
    tensors = Tensors(s, _tensor_specs(spec, len(row_req), T))
    return Workload(spec, L, r, cap, cache_start, T, row_req, row_pos,
                    prompt.numpy(), offsets, draft.numpy(), argmax.numpy(), tensors)


def draft_tensors(w: Workload) -> Tensors:
    """Inputs of the draft layer (the same on-demand set as the target's): the
    draft pool (latent + indexer key), the 6-row window of draft-layer KV to
    write back, and the per-step queries."""
    return w.tensors


def stochastic_inputs(seed: int, B: int, K: int, V: int, temperature: float = 1.0, noise: float = 0.5):
    """Synthetic inputs of rejection-sampling acceptance: target probabilities
    p [B, K+1, V] = softmax of N(0, 1) logits / temperature, draft probabilities
    q [B, K, V] = softmax of the same logits plus N(0, noise^2) (a draft that
    roughly follows the target), draft tokens drawn from q by inverse CDF with
    the generator's own uniforms, and the uniforms of the accept tests and of
    the draws.  Returns numpy arrays (draft, q, p, u_accept, u_sample)."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, _key("stochastic"), B, K, V])))
    logits = g.standard_normal((B, K + 1, V)) / temperature
    p = np.exp(logits - logits.max(axis=2, keepdims=True))
    p /= p.sum(axis=2, keepdims=True)
    dl = logits[:, :K] + noise * g.standard_normal((B, K, V))
    q = np.exp(dl - dl.max(axis=2, keepdims=True))
    q /= q.sum(axis=2, keepdims=True)
    cq = np.cumsum(q, axis=2)
    ud = g.random((B, K))
    draft = np.minimum((cq < (ud * cq[:, :, -1])[:, :, None]).sum(axis=2), V - 1).astype(np.int64)
    return (draft, q.astype(np.float32), p.astype(np.float32), g.random((B, K)).astype(np.float32),
            g.random(B).astype(np.float32))


def stochastic_inputs_device(seed: int, B: int, K: int, V: int, device, temperature: float = 1.0,
                             noise: float = 0.5):
    """The recipe of stochastic_inputs drawn on the device with torch's seeded
    CUDA generator (for vocabulary-sized batches whose host generation would
    take longer than the timing; not bit-identical to the host draw).  Draft
    tokens are drawn from q with torch.multinomial.  Returns device tensors
    (draft, q, p, u_accept, u_sample)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000003 + _key("stochastic") % 1000003)
    logits = torch.randn(B, K + 1, V, generator=g, device=device) / temperature
    p = torch.softmax(logits, dim=2)
    q = torch.softmax(logits[:, :K] + noise * torch.randn(B, K, V, generator=g, device=device), dim=2)
    draft = torch.multinomial(q.reshape(B * K, V), 1, generator=g).reshape(B, K).to(torch.int64)
    return (draft, q.contiguous(), p.contiguous(), torch.rand(B, K, generator=g, device=device),
            torch.rand(B, generator=g, device=device))


def layer_name(name: str, layer: int) -> str:
    """Name of a per-layer input: the first layer keeps the plain name."""
    return name if layer == 0 else f"{name}@{layer}"


def add_layers(w: Workload, n_layers: int) -> Workload:
    """Inputs of layers 1..n_layers-1 of a multi-layer verify (the same shapes as
    layer 0, their own streams): indexer queries, weights and keys, latent pool
    and MLA queries."""
    for l in range(1, n_layers):
        for base in ("q_idx", "w_idx", "k_idx", "latent", "q_mla"):
            w.tensors.specs[layer_name(base, l)] = w.tensors.specs[base]
    return w


def add_draft_extend(w: Workload) -> Workload:
    """Inputs of draft_extend's attention over the window rows in the draft layer:
    indexer queries and weights and MLA queries of each of the K+1 rows."""
    spec = w.spec
    B, W = spec.B, spec.K + 1
    std_i = 1.0 / math.sqrt(spec.D_I) if spec.scaled_normal else 1.0
    std_l = 1.0 / math.sqrt(576.0) if spec.scaled_normal else 1.0
    lat = torch.float32 if spec.latent_f32 else torch.bfloat16
    w.tensors.specs.update({
        "x_q_idx": TensorSpec((B * W, spec.H_I, spec.D_I), "normal", std_i, torch.float32),
        "x_w_idx": TensorSpec((B * W, spec.H_I), "uniform", 1.0, torch.float32),
        "x_q_mla": TensorSpec((B * W, spec.H_Q, 576), "normal", std_l, lat),
    })
    return w
