"""Seeded synthetic inputs for paged relative-bias GQA attention.

This module holds the workload shapes and the random-input recipe only: it contains
none of the attention arithmetic, so the CUDA path and the fp64 oracle can both be fed
from it without sharing any of the method.

Recipe (every tensor is drawn from a seeded ``torch.Generator``):

* Q, K, V: bf16, standard normal.
* ``rel_logits``: fp32, normal with standard deviation 0.5, shape ``[tokens, Hq, E]``.
* K/V pools: ``[num_pages, Hkv, P, D]``.  A sequence of length L owns ``ceil(L/P)``
  pages, placed at random positions of the pool; at least 10 % extra pages are
  allocated and filled with NaN, so any read of a page that is not the sequence's own
  shows up as a NaN in the output.
* block table ``[B, max_pages]`` int32: positional (entry j is the page of keys
  ``j*P .. j*P+P-1``); entries past a sequence's own pages hold ``num_pages + 7``, an
  id outside the pool, since the kernel must never read them ("Inkling attn backend
  cleanup fake registry", TensorRT-LLM PR #17860: seq_len bounds every access).
* ``seq_lens`` int32: KV length including this step's new tokens; ``cu_q_lens`` int32
  prefix sums of the new-token counts.

The five workloads are the shapes of the model described in "Support Inkling-NVFP4
model" (TensorRT-LLM PR #17062), section "Architecture": local layers with a 512-key
window and 16 KV heads, global full-causal layers with 8 KV heads, 64 query heads,
head_dim 128.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import numpy as np
import torch

TAIL_PAGE_OFFSET = 7  # block-table tail entries are num_pages + 7: never a real page


@dataclasses.dataclass
class Problem:
    """One call's worth of inputs (device or host tensors) plus its scalars."""

    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    rel_extent: int
    window: int
    sm_scale: float
    q_lens: List[int]
    seq_lens_list: List[int]
    q: torch.Tensor            # [total_q, Hq, D] bf16
    k_cache: torch.Tensor      # [num_pages, Hkv, P, D] bf16
    v_cache: torch.Tensor      # [num_pages, Hkv, P, D] bf16
    block_table: torch.Tensor  # [B, max_pages] int32
    seq_lens: torch.Tensor     # [B] int32
    cu_q_lens: torch.Tensor    # [B + 1] int32
    rel_logits: torch.Tensor   # [total_q, Hq, E] fp32 (empty when the bias is low-rank)
    seed: int = 0
    r: Optional[torch.Tensor] = None           # low-rank bias: [total_q, Hq, d_rel] bf16
    rel_proj_t: Optional[torch.Tensor] = None  # low-rank bias: [E, d_rel] bf16

    @property
    def num_seqs(self) -> int:
        return len(self.seq_lens_list)

    @property
    def total_q(self) -> int:
        return int(sum(self.q_lens))

    @property
    def num_pages(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def max_q_len(self) -> int:
        return int(max(self.q_lens)) if self.q_lens else 0

    @property
    def is_decode(self) -> bool:
        return all(n == 1 for n in self.q_lens)

    def visible_counts(self) -> List[List[int]]:
        """Per sequence, the number of visible keys of each new token (index bookkeeping)."""
        res = []
        for n, L in zip(self.q_lens, self.seq_lens_list):
            pos = np.arange(L - n, L, dtype=np.int64)
            lo = np.zeros_like(pos) if self.window <= 0 else np.maximum(0, pos - self.window + 1)
            res.append((pos - lo + 1).tolist())
        return res

    def to(self, device) -> "Problem":
        fields = {f.name: getattr(self, f.name) for f in dataclasses.fields(self)}
        for k, v in list(fields.items()):
            if isinstance(v, torch.Tensor):
                fields[k] = v.to(device)
        return Problem(**fields)

    def oracle_kwargs(self) -> Dict:
        """The inputs as numpy arrays in the form the fp64 oracle takes (bf16 as bits)."""
        def bits(t):
            return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
        return dict(num_q_heads=self.num_q_heads, num_kv_heads=self.num_kv_heads,
                    head_dim=self.head_dim, page_size=self.page_size,
                    rel_extent=self.rel_extent, window=self.window, sm_scale=self.sm_scale,
                    cu_q=self.cu_q_lens.cpu().numpy(), seq_lens=self.seq_lens.cpu().numpy(),
                    q_bits=bits(self.q), k_bits=bits(self.k_cache), v_bits=bits(self.v_cache),
                    block_table=self.block_table.cpu().numpy(),
                    rel=self.rel_logits.detach().float().cpu().numpy())

    def lowrank_bits(self):
        """(r bits, proj_t bits) of a low-rank-bias problem, as the oracle takes them."""
        def bits(t):
            return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
        return bits(self.r), bits(self.rel_proj_t)


def _randn(shape, gen, device, dtype, std=1.0):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def make_problem(*, num_q_heads: int, num_kv_heads: int, head_dim: int, page_size: int,
                 rel_extent: int, window: int, q_lens: List[int], seq_lens: List[int],
                 seed: int, device="cpu", sm_scale: Optional[float] = None,
                 extra_page_frac: float = 0.1, max_pages: Optional[int] = None,
                 rel_std: float = 0.5, nan_spare_pages: bool = True,
                 bias_dtype=torch.float32, lowrank_d: Optional[int] = None) -> Problem:
    """Build a seeded problem.  ``q_lens[b]`` new tokens are the last of ``seq_lens[b]``.

    ``bias_dtype=torch.bfloat16`` rounds the same seeded bias to bf16 (the input of the
    bf16-bias prefill); the oracle then reads those rounded values.

    ``lowrank_d`` gives the bias in low-rank form instead: r ``[T, Hq, d]`` bf16 N(0,1) and
    the transposed projection ``[E, d]`` bf16 N(0, rel_std^2 / d), so that the bias they
    define has standard deviation ``rel_std``; ``rel_logits`` is then empty."""
    assert len(q_lens) == len(seq_lens)
    for n, L in zip(q_lens, seq_lens):
        assert 0 <= n <= L or (L == 0 and n == 0)
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    host_gen = torch.Generator()
    host_gen.manual_seed(seed + 1_000_003)
    B = len(seq_lens)
    pages_per_seq = [(L + page_size - 1) // page_size for L in seq_lens]
    used = sum(pages_per_seq)
    spare = max(1, int(math.ceil(extra_page_frac * used)))
    num_pages = used + spare
    width = max(pages_per_seq + [1]) if max_pages is None else max_pages
    assert width >= max(pages_per_seq + [0])
    perm = torch.randperm(num_pages, generator=host_gen)
    bt = torch.full((B, width), num_pages + TAIL_PAGE_OFFSET, dtype=torch.int32)
    cur = 0
    for b, npg in enumerate(pages_per_seq):
        bt[b, :npg] = perm[cur:cur + npg].to(torch.int32)
        cur += npg
    spare_ids = perm[cur:]
    pool_shape = (num_pages, num_kv_heads, page_size, head_dim)
    k_cache = _randn(pool_shape, gen, device, torch.bfloat16)
    v_cache = _randn(pool_shape, gen, device, torch.bfloat16)
    if nan_spare_pages and spare_ids.numel():
        idx = spare_ids.to(device)
        k_cache[idx] = float("nan")
        v_cache[idx] = float("nan")
    total_q = int(sum(q_lens))
    q = _randn((total_q, num_q_heads, head_dim), gen, device, torch.bfloat16)
    r = proj_t = None
    if lowrank_d is None:
        rel = _randn((total_q, num_q_heads, rel_extent), gen, device, bias_dtype, std=rel_std)
    else:
        rel = torch.empty(0, dtype=torch.float32, device=device)
        r = _randn((total_q, num_q_heads, lowrank_d), gen, device, torch.bfloat16)
        proj_t = _randn((rel_extent, lowrank_d), gen, device, torch.bfloat16, std=rel_std / math.sqrt(lowrank_d))
    cu = torch.zeros(B + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(q_lens, dtype=torch.int64), 0).to(torch.int32)
    return Problem(num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                   page_size=page_size, rel_extent=rel_extent, window=window,
                   sm_scale=(1.0 / math.sqrt(head_dim)) if sm_scale is None else sm_scale,
                   q_lens=list(q_lens), seq_lens_list=list(seq_lens), q=q,
                   k_cache=k_cache, v_cache=v_cache, block_table=bt.to(device),
                   seq_lens=torch.tensor(seq_lens, dtype=torch.int32, device=device),
                   cu_q_lens=cu.to(device), rel_logits=rel, seed=seed, r=r, rel_proj_t=proj_t)


def _uniform_lengths(n, lo, hi, seed):
    g = torch.Generator()
    g.manual_seed(seed)
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


def _log_uniform_lengths(n, lo, hi, seed):
    g = torch.Generator()
    g.manual_seed(seed)
    u = torch.rand(n, generator=g, dtype=torch.float64)
    return [int(round(math.exp(math.log(lo) + x * (math.log(hi) - math.log(lo))))) for x in u.tolist()]


# Layer geometries of the model ("Architecture" section of PR #17062).
SWA_LAYER = dict(num_q_heads=64, num_kv_heads=16, head_dim=128, window=512, rel_extent=512)
GLOBAL_LAYER = dict(num_q_heads=64, num_kv_heads=8, head_dim=128, window=-1, rel_extent=4096)


def swa_prefill_tiny(device="cpu", seed=0) -> Problem:
    """1 x 1024 tokens, 8 query heads over 2 KV heads, D 64, window 512, E 512, P 16."""
    return make_problem(num_q_heads=8, num_kv_heads=2, head_dim=64, page_size=16,
                        rel_extent=512, window=512, q_lens=[1024], seq_lens=[1024],
                        seed=seed, device=device)


def swa_decode(device="cpu", seed=2, batch=64) -> Problem:
    """SWA-layer decode: batch 64, contexts U{1024..8192}, page 64."""
    L = _uniform_lengths(batch, 1024, 8192, seed)
    return make_problem(**SWA_LAYER, page_size=64, q_lens=[1] * batch, seq_lens=L,
                        seed=seed, device=device)


def global_decode(device="cpu", seed=3, batch=32) -> Problem:
    """Global-layer decode: batch 32, contexts U{8192..32768}, E 4096 (clamped), page 64."""
    L = _uniform_lengths(batch, 8192, 32768, seed)
    return make_problem(**GLOBAL_LAYER, page_size=64, q_lens=[1] * batch, seq_lens=L,
                        seed=seed, device=device)


def global_prefill(device="cpu", seed=4, batch=4, tokens=8192, bias_dtype=torch.float32) -> Problem:
    """Global-layer prefill: 4 x 8192 tokens, full causal, E 4096, page 64."""
    return make_problem(**GLOBAL_LAYER, page_size=64, q_lens=[tokens] * batch,
                        seq_lens=[tokens] * batch, seed=seed, device=device, bias_dtype=bias_dtype)


# Rank of the low-rank bias workloads: the pages do not give d_rel; 64 is a plausible size
# for a per-head relative-position code.
LOWRANK_D = 64


def global_prefill_lowrank(device="cpu", seed=4, batch=4, tokens=8192, d_rel=LOWRANK_D) -> Problem:
    """Global-layer prefill with the bias in low-rank form: 4 x 8192 tokens, E 4096, d_rel 64."""
    return make_problem(**GLOBAL_LAYER, page_size=64, q_lens=[tokens] * batch,
                        seq_lens=[tokens] * batch, seed=seed, device=device, lowrank_d=d_rel)


def mixed_layer(kind: str, layer: int, device="cpu", seed=5,
                n_prefill=8, prefill_tokens=2048, n_decode=128):
    """One layer of the mixed serving batch: (prefill problem, decode problem).

    5 SWA layers + 1 global layer; per layer one prefill call over 8 x 2048-token
    prompts and one decode call over 128 requests with log-uniform contexts 512..16384.
    Every layer has its own pool.
    """
    geo = SWA_LAYER if kind == "swa" else GLOBAL_LAYER
    base = seed * 1000 + layer * 10
    pre = make_problem(**geo, page_size=64, q_lens=[prefill_tokens] * n_prefill,
                       seq_lens=[prefill_tokens] * n_prefill, seed=base, device=device)
    L = _log_uniform_lengths(n_decode, 512, 16384, seed)
    dec = make_problem(**geo, page_size=64, q_lens=[1] * n_decode, seq_lens=L,
                       seed=base + 1, device=device)
    return pre, dec


MIXED_STACK = ["swa", "swa", "swa", "swa", "swa", "global"]

WORKLOADS = {
    "swa_prefill_tiny": swa_prefill_tiny,
    "swa_decode": swa_decode,
    "global_decode": global_decode,
    "global_prefill": global_prefill,
}


@dataclasses.dataclass
class KvStep:
    """One call of the K/V short convolution and paged write: the step's raw K/V rows,
    the filters, the carried state, and the paged pools they are written into."""

    num_kv_heads: int
    head_dim: int
    page_size: int
    kernel_size: int
    q_lens: List[int]
    seq_lens_list: List[int]
    k_new: torch.Tensor        # [T, Hkv, D] bf16
    v_new: torch.Tensor
    w_k: torch.Tensor          # [Hkv, D, ks] fp32
    w_v: torch.Tensor
    state_k: torch.Tensor      # [B, ks-1, Hkv, D] bf16, oldest row first
    state_v: torch.Tensor
    k_cache: torch.Tensor      # [num_pages, Hkv, P, D] bf16
    v_cache: torch.Tensor
    block_table: torch.Tensor  # [B, max_pages] int32
    seq_lens: torch.Tensor     # [B] int32
    cu_q_lens: torch.Tensor    # [B + 1] int32

    @property
    def num_seqs(self) -> int:
        return len(self.seq_lens_list)

    @property
    def total_q(self) -> int:
        return int(sum(self.q_lens))

    @property
    def num_pages(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])

    def oracle_kwargs(self) -> Dict:
        def bits(t):
            return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
        return dict(k_new_bits=bits(self.k_new), v_new_bits=bits(self.v_new),
                    cu_q=self.cu_q_lens.cpu().numpy(), seq_lens=self.seq_lens.cpu().numpy(),
                    block_table=self.block_table.cpu().numpy(), page_size=self.page_size,
                    w_k=self.w_k.double().cpu().numpy(), w_v=self.w_v.double().cpu().numpy(),
                    ks=self.kernel_size, state_k_bits=bits(self.state_k), state_v_bits=bits(self.state_v),
                    k_cache_bits=bits(self.k_cache), v_cache_bits=bits(self.v_cache))


def make_kv_step(*, num_kv_heads: int, head_dim: int, page_size: int, kernel_size: int,
                 q_lens: List[int], seq_lens: List[int], seed: int, device="cpu",
                 extra_page_frac: float = 0.1) -> KvStep:
    """Seeded inputs of one K/V write.  Recipe: new K/V rows and the pools' old contents
    bf16 N(0,1) (spare pages NaN, so a write to a page that is not the request's own
    is visible); filters fp32 N(0, 1/ks); carried state bf16 N(0,1), except that a
    request whose step holds its whole history (n_b == L_b) starts from zero rows;
    pages placed at random, block-table tails num_pages + 7 as in ``make_problem``."""
    assert len(q_lens) == len(seq_lens)
    for n, L in zip(q_lens, seq_lens):
        assert 0 <= n <= L
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    host_gen = torch.Generator()
    host_gen.manual_seed(seed + 2_000_003)
    B, Hkv, D, P, ks = len(seq_lens), num_kv_heads, head_dim, page_size, kernel_size
    pages_per_seq = [(L + P - 1) // P for L in seq_lens]
    used = sum(pages_per_seq)
    num_pages = used + max(1, int(math.ceil(extra_page_frac * used)))
    width = max(pages_per_seq + [1])
    perm = torch.randperm(num_pages, generator=host_gen)
    bt = torch.full((B, width), num_pages + TAIL_PAGE_OFFSET, dtype=torch.int32)
    cur = 0
    for b, npg in enumerate(pages_per_seq):
        bt[b, :npg] = perm[cur:cur + npg].to(torch.int32)
        cur += npg
    spare_ids = perm[cur:].to(device)
    pool = (num_pages, Hkv, P, D)
    k_cache = _randn(pool, gen, device, torch.bfloat16)
    v_cache = _randn(pool, gen, device, torch.bfloat16)
    if spare_ids.numel():
        k_cache[spare_ids] = float("nan")
        v_cache[spare_ids] = float("nan")
    T = int(sum(q_lens))
    k_new = _randn((T, Hkv, D), gen, device, torch.bfloat16)
    v_new = _randn((T, Hkv, D), gen, device, torch.bfloat16)
    w_k = _randn((Hkv, D, ks), gen, device, torch.float32, std=1.0 / math.sqrt(ks))
    w_v = _randn((Hkv, D, ks), gen, device, torch.float32, std=1.0 / math.sqrt(ks))
    state_k = _randn((B, ks - 1, Hkv, D), gen, device, torch.bfloat16)
    state_v = _randn((B, ks - 1, Hkv, D), gen, device, torch.bfloat16)
    fresh = [b for b, (n, L) in enumerate(zip(q_lens, seq_lens)) if n == L]
    if fresh and ks > 1:
        idx = torch.tensor(fresh, device=device)
        state_k[idx] = 0
        state_v[idx] = 0
    cu = torch.zeros(B + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(q_lens, dtype=torch.int64), 0).to(torch.int32)
    return KvStep(num_kv_heads=Hkv, head_dim=D, page_size=P, kernel_size=ks, q_lens=list(q_lens),
                  seq_lens_list=list(seq_lens), k_new=k_new, v_new=v_new, w_k=w_k, w_v=w_v,
                  state_k=state_k, state_v=state_v, k_cache=k_cache, v_cache=v_cache,
                  block_table=bt.to(device), seq_lens=torch.tensor(seq_lens, dtype=torch.int32, device=device),
                  cu_q_lens=cu.to(device))


def kv_step_for(prob: Problem, kernel_size: int, seed: int) -> KvStep:
    """K/V write inputs for an attention problem's step, writing into that problem's own pools
    (its cache, block table, lengths and query offsets are shared, not copied): the new rows,
    filters and carried state are drawn as in ``make_kv_step``."""
    dev = prob.k_cache.device
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    T, B, Hkv, D, ks = prob.total_q, prob.num_seqs, prob.num_kv_heads, prob.head_dim, kernel_size
    k_new = _randn((T, Hkv, D), gen, dev, torch.bfloat16)
    v_new = _randn((T, Hkv, D), gen, dev, torch.bfloat16)
    w_k = _randn((Hkv, D, ks), gen, dev, torch.float32, std=1.0 / math.sqrt(ks))
    w_v = _randn((Hkv, D, ks), gen, dev, torch.float32, std=1.0 / math.sqrt(ks))
    state_k = _randn((B, ks - 1, Hkv, D), gen, dev, torch.bfloat16)
    state_v = _randn((B, ks - 1, Hkv, D), gen, dev, torch.bfloat16)
    fresh = [b for b, (n, L) in enumerate(zip(prob.q_lens, prob.seq_lens_list)) if n == L]
    if fresh and ks > 1:
        idx = torch.tensor(fresh, device=dev)
        state_k[idx] = 0
        state_v[idx] = 0
    return KvStep(num_kv_heads=Hkv, head_dim=D, page_size=prob.page_size, kernel_size=ks, q_lens=list(prob.q_lens),
                  seq_lens_list=list(prob.seq_lens_list), k_new=k_new, v_new=v_new, w_k=w_k, w_v=w_v,
                  state_k=state_k, state_v=state_v, k_cache=prob.k_cache, v_cache=prob.v_cache,
                  block_table=prob.block_table, seq_lens=prob.seq_lens, cu_q_lens=prob.cu_q_lens)


# Short-convolution kernel size of the K/V write workloads: the pages give none; 4 is the
# usual width of a causal short convolution in hybrid models.
KV_CONV_KERNEL = 4


def kv_prefill_global(device="cpu", seed=6, batch=4, tokens=8192) -> KvStep:
    """K/V write of a global-layer prefill: 4 fresh prompts of 8192 tokens, 8 KV heads."""
    return make_kv_step(num_kv_heads=GLOBAL_LAYER["num_kv_heads"], head_dim=128, page_size=64,
                        kernel_size=KV_CONV_KERNEL, q_lens=[tokens] * batch, seq_lens=[tokens] * batch,
                        seed=seed, device=device)


def kv_decode_swa(device="cpu", seed=7, batch=64) -> KvStep:
    """K/V write of an SWA-layer decode step: 64 requests, contexts U{1024..8192}."""
    L = _uniform_lengths(batch, 1024, 8192, seed)
    return make_kv_step(num_kv_heads=SWA_LAYER["num_kv_heads"], head_dim=128, page_size=64,
                        kernel_size=KV_CONV_KERNEL, q_lens=[1] * batch, seq_lens=L, seed=seed, device=device)


def sample_rows(prob: Problem, per_seq: int, seed: int) -> np.ndarray:
    """A seeded sample of (packed row, head) pairs for oracle checks on big problems.

    Per sequence: at least ``per_seq`` distinct pairs (every pair when the sequence has
    fewer), always including the rows at positions 0, 1, 510, 511, 512, 4094, 4095, 4096
    and L-1 where they exist and the page-boundary rows, each on the first head of every
    KV group; the rest is drawn uniformly without replacement.
    Returns an int32 array ``[n, 2]`` of (t, h), sorted.
    """
    rng = np.random.default_rng(seed)
    out = []
    cu = prob.cu_q_lens.cpu().numpy()
    Hq = prob.num_q_heads
    step = max(1, Hq // prob.num_kv_heads)
    for b, (n, L) in enumerate(zip(prob.q_lens, prob.seq_lens_list)):
        if n == 0:
            continue
        first = L - n
        want = {0, 1, 510, 511, 512, 4094, 4095, 4096, L - 1,
                prob.page_size - 1, prob.page_size, 2 * prob.page_size - 1}
        pos = [p for p in want if first <= p < L]
        fixed = {(p - first) * Hq + h for p in pos for h in range(0, Hq, step)}
        k = min(n * Hq, max(per_seq, len(fixed))) - len(fixed)
        pool = np.setdiff1d(np.arange(n * Hq, dtype=np.int64), np.fromiter(fixed, np.int64, len(fixed)))
        pick = np.concatenate([np.fromiter(fixed, np.int64, len(fixed)),
                               rng.choice(pool, size=k, replace=False)])
        for x in np.sort(pick).tolist():
            out.append((int(cu[b]) + x // Hq, x % Hq))
    arr = np.asarray(out, dtype=np.int32).reshape(-1, 2)
    return arr


def rows_per_sequence(prob: Problem, rows: np.ndarray) -> List[int]:
    """How many sampled rows fall in each sequence (for the parity tests' printout)."""
    cu = prob.cu_q_lens.cpu().numpy()
    t = np.sort(rows[:, 0]) if rows.size else np.zeros(0, np.int32)
    edges = np.searchsorted(t, cu, side="left")
    return np.diff(edges).tolist()
