"""Seeded synthetic inputs for paged-KV decode attention.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no softmax, no prefix sums, no slot arithmetic beyond the
page assignment it invents).  Both the CPU oracle (``oracle/``) and the CUDA
path (tests, ``bench.py``) take their inputs from here, so the two sides see
bit-identical data.

Workloads are shaped like the decode batches the engine's commit log describes
(AstrAI, "astrai/inference/core/cache.py" page: 4-D KV storage
``[n_layers, size, n_kv_heads, head_dim]``, a request-to-token table, per-step
``seq_lens``).  Every value is synthetic; no dataset is involved.

Recipe (shared by all named workloads):
  * values: standard normal fp32 drawn with numpy PCG64 in fixed 4 Mi-element
    chunks (chunk i seeded by ``SeedSequence(seed).spawn``), cast to bf16 with
    round-to-nearest-even;
  * pages: the pool's pages are a random permutation; request b receives a
    contiguous run of that permutation, so its pages are scattered;
  * ``req_pool_indices``: a random choice of table rows out of
    ``max_reqs = 2 * batch``; unused table entries hold -1;
  * ``seq_lens`` are the cached lengths *before* a decode step; the pool has
    room for ``steps`` more tokens per request.
"""
from __future__ import annotations

import dataclasses
import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

INDEX_PAGE_TABLE = 0
INDEX_FLAT = 1

_CHUNK = 1 << 22  # elements per independently seeded chunk


@dataclasses.dataclass
class DecodeProblem:
    """One batch of cached decode state (all tensors on the CPU)."""

    name: str
    batch: int
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    page_size: int
    index_mode: int
    pool_slots: int
    max_reqs: int
    max_pages_per_req: int
    steps: int                      # steady steps the pool has room for
    seq_lens: torch.Tensor          # int32 [B], cached tokens before the step
    req_pool_indices: torch.Tensor  # int32 [B]
    page_table: torch.Tensor        # int32 [max_reqs, max_pages_per_req]
    k_pool: torch.Tensor            # bf16 [NL, pool_slots, Hkv, D]
    v_pool: torch.Tensor            # bf16 [NL, pool_slots, Hkv, D]
    scale: float                    # softmax scale, an fp32-representable value
    seed: int
    shared_prefix_pages: int = 0    # leading table entries every request shares

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def max_total_tokens(self) -> int:
        return int(self.batch * self.max_pages_per_req * self.page_size)


def _normal_f32(n: int, seed: int, threads: int = 0) -> np.ndarray:
    """n standard normals, deterministic for a seed whatever the thread count."""
    out = np.empty(n, dtype=np.float32)
    n_chunks = max(1, (n + _CHUNK - 1) // _CHUNK)
    children = np.random.SeedSequence(seed).spawn(n_chunks)

    def fill(i):
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        np.random.default_rng(children[i]).standard_normal(out=out[lo:hi], dtype=np.float32)

    workers = threads or min(16, (torch.get_num_threads() or 1) * 2)
    if n_chunks == 1:
        fill(0)
    else:
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(fill, range(n_chunks)))
    return out


def normal_bf16(shape, seed: int) -> torch.Tensor:
    """Standard-normal bf16 tensor (fp32 draw, round-to-nearest-even cast)."""
    n = int(np.prod(shape))
    return torch.from_numpy(_normal_f32(n, seed)).view(*shape).to(torch.bfloat16)


def _sub(seed: int, k: int) -> int:
    return seed * 64 + k


def make_problem(
    name: str = "custom",
    *,
    batch: int,
    n_layers: int,
    n_q_heads: int,
    n_kv_heads: int,
    head_dim: int,
    page_size: int,
    seq_lens,
    steps: int = 0,
    pool_factor: float = 2.0,
    pool_pages: int | None = None,
    index_mode: int | None = None,
    outlier_frac: float = 0.0,
    outlier_scale: float = 8.0,
    scale: float | None = None,
    seed: int = 20260000,
    fill_unused: bool = True,
    shared_prefix_pages: int = 0,
) -> DecodeProblem:
    """Build one decode problem.

    ``seq_lens`` is a list of cached lengths.  Flat mode (token-level
    ``kv_indices``) is used when ``page_size == 1`` unless ``index_mode`` says
    otherwise; then ``page_table`` is the request-to-token table.
    ``shared_prefix_pages`` > 0: every request's first that many table
    entries are the same physical pages (request 0's), stored once.
    """
    seq = [int(x) for x in seq_lens]
    assert len(seq) == batch
    P = page_size
    if index_mode is None:
        index_mode = INDEX_FLAT if P == 1 else INDEX_PAGE_TABLE
    pages_per_req = [max(1, math.ceil((L + steps) / P)) for L in seq]
    sp = shared_prefix_pages
    assert all(n > sp for n in pages_per_req) or sp == 0, "a request must own a page past the prefix"
    need = sum(pages_per_req) - sp * (batch - 1)
    n_pages = pool_pages if pool_pages is not None else max(need, int(math.ceil(need * pool_factor)))
    assert n_pages >= need, "pool too small"
    pool_slots = n_pages * P
    max_pages = max(pages_per_req)
    max_reqs = 2 * batch

    g = torch.Generator().manual_seed(_sub(seed, 1))
    perm = torch.randperm(n_pages, generator=g).to(torch.int32)
    rows = torch.randperm(max_reqs, generator=g)[:batch].to(torch.int32)
    table = torch.full((max_reqs, max_pages), -1, dtype=torch.int32)
    off = 0
    for b in range(batch):
        n = pages_per_req[b]
        if b > 0 and sp:
            table[rows[b], :sp] = table[rows[0], :sp]
            table[rows[b], sp:n] = perm[off:off + n - sp]
            off += n - sp
        else:
            table[rows[b], :n] = perm[off:off + n]
            off += n

    shape = (n_layers, pool_slots, n_kv_heads, head_dim)
    if fill_unused:
        kf = torch.from_numpy(_normal_f32(int(np.prod(shape)), _sub(seed, 2))).view(*shape)
        vf = torch.from_numpy(_normal_f32(int(np.prod(shape)), _sub(seed, 3))).view(*shape)
    else:
        kf = torch.zeros(shape)
        vf = torch.zeros(shape)
    if outlier_frac > 0:
        # Outlier key rows: a seeded share of the token positions in use, all
        # KV heads of that slot, scaled before the bf16 cast.
        go = torch.Generator().manual_seed(_sub(seed, 4))
        used = []
        for b in range(batch):
            pages = table[rows[b], :pages_per_req[b]].to(torch.int64)
            slots = (pages[:, None] * P + torch.arange(P)[None, :]).reshape(-1)[: seq[b]]
            used.append(slots)
        used = torch.cat(used)
        n_out = max(1, int(round(outlier_frac * used.numel())))
        pick = used[torch.randperm(used.numel(), generator=go)[:n_out]]
        kf[:, pick] *= outlier_scale
    k_pool = kf.to(torch.bfloat16)
    del kf
    v_pool = vf.to(torch.bfloat16)
    del vf
    if scale is None:
        scale = float(np.float32(1.0 / math.sqrt(head_dim)))
    return DecodeProblem(
        name=name, batch=batch, n_layers=n_layers, n_q_heads=n_q_heads,
        n_kv_heads=n_kv_heads, head_dim=head_dim, page_size=P, index_mode=index_mode,
        pool_slots=pool_slots, max_reqs=max_reqs, max_pages_per_req=max_pages,
        steps=steps, seq_lens=torch.tensor(seq, dtype=torch.int32),
        req_pool_indices=rows, page_table=table, k_pool=k_pool, v_pool=v_pool,
        scale=scale, seed=seed, shared_prefix_pages=shared_prefix_pages,
    )


def step_inputs(p: DecodeProblem, step: int, layers=None):
    """Per-step inputs: q [NL,B,Hq,D], k_new and v_new [NL,B,Hkv,D] (bf16)."""
    NL = p.n_layers if layers is None else layers
    s = _sub(p.seed, 16 + 3 * step)
    q = normal_bf16((NL, p.batch, p.n_q_heads, p.head_dim), s)
    k = normal_bf16((NL, p.batch, p.n_kv_heads, p.head_dim), s + 1)
    v = normal_bf16((NL, p.batch, p.n_kv_heads, p.head_dim), s + 2)
    return q, k, v


# --------------------------------------------------------------------------
# Named workloads.  Sizes follow the decode batches the engine's pages describe;
# ``shrink`` gives the same recipe at sizes a CPU oracle finishes in seconds.
# --------------------------------------------------------------------------

WORKLOADS = ("single_d64", "gqa4_b4_paged", "gqa4_b16_flat_skewed",
             "gqa4_long_65536", "gqa8_graph_sweep", "shared_prefix_b32")


def _uniform_lens(n, lo, hi, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


def _loguniform_lens(n, hi, seed):
    g = torch.Generator().manual_seed(seed)
    u = torch.rand(n, generator=g, dtype=torch.float64)
    return [int(min(hi, max(1, round(math.exp(x * math.log(hi)))))) for x in u.tolist()]


def workload(name: str, *, batch: int | None = None, n_layers: int | None = None,
             steps: int = 0, shrink: int = 1, seed: int | None = None,
             fill_unused: bool = True) -> DecodeProblem:
    """The five decode workloads.

    single_d64          B=1, 1 layer, 8/2 heads, D=64, P=16, L=128 in a
                        64-page permuted pool, scale 1/8.
    gqa4_b4_paged       B=4, 24 layers, 32/8 heads, D=128, P=16,
                        L ~ U{512..2048}, pool 2x the pages needed.
    gqa4_b16_flat_skewed B=16, 24 layers, 32/8, D=128, P=1 (token-level
                        kv_indices), L log-uniform in [1, 8192], pool 2x.
    gqa4_long_65536     B=1 or 4, 1 layer, 32/8, D=128, P=16, L=65536,
                        1% of key rows scaled x8.
    gqa8_graph_sweep    B in {1,4,8,16,32,64}, 24 layers, 16/2, D=128, P=16,
                        L ~ U{1024..4096}.
    shared_prefix_b32   B=32, 24 layers, 32/8, D=128, P=16: every request's
                        first 4096 tokens are the same 256 pages (stored
                        once), then 64..192 tokens of its own.

    ``shrink`` > 1 divides lengths (and layers, to at most 2) for the
    oracle-sized variants of the same recipe.
    """
    idx = WORKLOADS.index(name) + 1
    seed = 20260000 + idx if seed is None else seed
    if name == "single_d64":
        B = batch or 1
        return make_problem(name, batch=B, n_layers=n_layers or 1, n_q_heads=8, n_kv_heads=2,
                            head_dim=64, page_size=16, seq_lens=[128] * B, steps=steps,
                            pool_pages=max(64, B * 8 + B * math.ceil(steps / 16) * 2),
                            scale=0.125, seed=seed, fill_unused=fill_unused)
    if name == "gqa4_b4_paged":
        B = batch or 4
        lens = _uniform_lens(B, max(1, 512 // shrink), max(1, 2048 // shrink), _sub(seed, 0))
        nl = n_layers or (24 if shrink == 1 else 2)
        return make_problem(name, batch=B, n_layers=nl, n_q_heads=32, n_kv_heads=8,
                            head_dim=128, page_size=16, seq_lens=lens, steps=steps,
                            seed=seed, fill_unused=fill_unused)
    if name == "gqa4_b16_flat_skewed":
        B = batch or 16
        lens = _loguniform_lens(B, max(1, 8192 // shrink), _sub(seed, 0))
        nl = n_layers or (24 if shrink == 1 else 2)
        return make_problem(name, batch=B, n_layers=nl, n_q_heads=32, n_kv_heads=8,
                            head_dim=128, page_size=1, seq_lens=lens, steps=steps,
                            seed=seed, fill_unused=fill_unused)
    if name == "gqa4_long_65536":
        B = batch or 1
        L = max(1, 65536 // shrink)
        return make_problem(name, batch=B, n_layers=n_layers or 1, n_q_heads=32, n_kv_heads=8,
                            head_dim=128, page_size=16, seq_lens=[L] * B, steps=steps,
                            pool_factor=1.0, outlier_frac=0.01, seed=seed,
                            fill_unused=fill_unused)
    if name == "shared_prefix_b32":
        B = batch or 32
        prefix = max(16, 4096 // shrink) // 16 * 16
        own = _uniform_lens(B, max(1, 64 // shrink), max(1, 192 // shrink), _sub(seed, 0))
        nl = n_layers or (24 if shrink == 1 else 2)
        return make_problem(name, batch=B, n_layers=nl, n_q_heads=32, n_kv_heads=8,
                            head_dim=128, page_size=16, seq_lens=[prefix + x for x in own],
                            steps=steps, pool_factor=1.0, seed=seed, fill_unused=fill_unused,
                            shared_prefix_pages=prefix // 16)
    if name == "gqa8_graph_sweep":
        B = batch or 16
        lens = _uniform_lens(B, max(1, 1024 // shrink), max(1, 4096 // shrink), _sub(seed, 0))
        nl = n_layers or (24 if shrink == 1 else 2)
        return make_problem(name, batch=B, n_layers=nl, n_q_heads=16, n_kv_heads=2,
                            head_dim=128, page_size=16, seq_lens=lens, steps=steps,
                            seed=seed, fill_unused=fill_unused)
    raise KeyError(name)


# --------------------------------------------------------------------------
# Extend (prefill) workload: requests whose newest tokens are a chunk of new
# positions on top of a cached prefix (the step before decode).
# --------------------------------------------------------------------------

EXTEND_WORKLOADS = ("extend_b4_chunk256", "extend_b1_prefix32k_chunk64")


def extend_workload(name: str, *, n_layers: int | None = None, shrink: int = 1,
                    seed: int | None = None):
    """Extend (prefill) workloads, 32/8 heads, D=128, P=16; the pool holds
    prefix + new tokens.  Returns the problem (its seq_lens count the new
    tokens) and the new-token counts.

    extend_b4_chunk256           B=4, 24 layers, cached prefixes ~ U{512..2048}
                                 (the paged decode workload's lengths), 256 new
                                 tokens per request.
    extend_b1_prefix32k_chunk64  B=1, 4 layers, a 32768-token cached prefix and
                                 64 new tokens (a short chunk on a long
                                 context); pool exactly the pages needed.

    ``shrink`` divides the lengths (and uses 2 layers)."""
    seed = (20260100 + EXTEND_WORKLOADS.index(name)) if seed is None else seed
    if name == "extend_b4_chunk256":
        B, chunk = 4, max(1, 256 // shrink)
        prefix = _uniform_lens(B, max(1, 512 // shrink), max(1, 2048 // shrink), _sub(seed, 0))
        nl = n_layers or (24 if shrink == 1 else 2)
        p = make_problem(name, batch=B, n_layers=nl, n_q_heads=32, n_kv_heads=8, head_dim=128,
                         page_size=16, seq_lens=[x + chunk for x in prefix], seed=seed)
        return p, [chunk] * B
    if name == "extend_b1_prefix32k_chunk64":
        chunk, prefix = max(1, 64 // shrink), max(1, 32768 // shrink)
        nl = n_layers or (4 if shrink == 1 else 2)
        p = make_problem(name, batch=1, n_layers=nl, n_q_heads=32, n_kv_heads=8, head_dim=128,
                         page_size=16, seq_lens=[prefix + chunk], pool_factor=1.0, seed=seed)
        return p, [chunk]
    raise KeyError(name)


def extend_inputs(p: DecodeProblem, qo_lens, layers=None):
    """Per-layer extend inputs: q [NL, T, Hq, D], k_new and v_new [NL, T, Hkv, D]
    (bf16), T = sum of the new-token counts."""
    NL = p.n_layers if layers is None else layers
    T = int(sum(qo_lens))
    s = _sub(p.seed, 40)
    q = normal_bf16((NL, T, p.n_q_heads, p.head_dim), s)
    k = normal_bf16((NL, T, p.n_kv_heads, p.head_dim), s + 1)
    v = normal_bf16((NL, T, p.n_kv_heads, p.head_dim), s + 2)
    return q, k, v
