"""Seeded synthetic inputs for the paged-KV compose and the ragged index plan.

This module is shared by the CPU oracle's tests, the GPU parity tests and the
benchmark.  It draws batch metadata (lengths, logical page tables, writer
ranks, chunk ownership) and KV row bytes from seeded generators.  It contains
none of the compose arithmetic: no spans, descriptors, inverses or locs are
computed here.  The only structure it knows is the scenario itself:

* a request's prefix occupies ``prefix_len / page_size`` logical pages and its
  current (extend) tokens occupy ``ceil(cur_len / page_size)`` pages;
* under the page-aligned in-seq split each current page has one writer rank,
  and that rank computes the KV rows of the page's tokens (commit log
  d63fbd4, "symm counting barrier + IPC gather" message: each current page is
  written by exactly one rank);
* the q tokens of the NSA indexer are cut into fixed-size chunks that are
  dealt to context-parallel ranks (commit log d63fbd4, "CPU-gap fixes"
  message: the ragged plan is keyed on ``cp_index``).

Workload shapes follow the five benchmark configurations of this project
(tiny, traced prefill, 78-layer loop, fp8 NSA, ragged plan), plus the NSA
index keys of the fp8 batch and the traced lengths on one-token pages.
Seeds: config k uses ``1000 + k``.  Streams are drawn in a fixed order from one
``numpy.random.Generator``.
"""
from __future__ import annotations

import dataclasses

import numpy as np

MLA_ROW_BYTES = 576 * 2  # 512 latent + 64 rope, bf16
NSA_FP8_ROW_BYTES = 512 + 4 * 4 + 64 * 2  # fp8 latent + 4 fp32 scales + 64 bf16 rope = 656


@dataclasses.dataclass
class ComposeBatch:
    """Batch metadata of one compose (host arrays, int32)."""

    name: str
    seed: int
    page_size: int
    cp_size: int
    num_pool_pages: int  # logical page ids live in [1, num_pool_pages); 0 is the dummy page
    row_bytes: int
    num_layers: int
    prefix_lens: np.ndarray  # [B] multiples of page_size
    cur_lens: np.ndarray  # [B]
    prefix_pages: np.ndarray  # CSR by request: prefix_lens[b] // page_size entries each
    cur_pages: np.ndarray  # CSR by request: ceil(cur_lens[b] / page_size) entries each
    writer: np.ndarray  # [C] writer rank of each current page, batch order
    row_kind: str  # "bf16" (N(0,1) values) or "bytes" (uniform random bytes)
    planes: tuple | None = None  # planar pages: bytes per token of each plane (sum = row_bytes)

    @property
    def B(self) -> int:
        return int(self.prefix_lens.shape[0])

    @property
    def T(self) -> int:
        return int(self.cur_lens.sum())

    @property
    def C(self) -> int:
        return int(self.cur_pages.shape[0])

    @property
    def num_prefix_pages(self) -> int:
        return int(self.prefix_pages.shape[0])

    @property
    def slab_pages(self) -> int:
        """Pages per owner slab of the pool (``ceil(P / cp)``)."""
        return -(-self.num_pool_pages // self.cp_size)

    @property
    def page_bytes(self) -> int:
        return self.page_size * self.row_bytes


def pages_per_len(n_tokens: np.ndarray, page_size: int) -> np.ndarray:
    """Pages needed to hold ``n_tokens`` tokens (ceil division)."""
    n = np.asarray(n_tokens, dtype=np.int64)
    return ((n + page_size - 1) // page_size).astype(np.int64)


def lognormal_split(rng: np.random.Generator, total: int, n: int, sigma: float = 1.0) -> np.ndarray:
    """Split ``total`` into ``n`` positive integers with lognormal weights.

    Weights exp(N(0, sigma^2)) are scaled to the total and rounded by largest
    remainder; every part is at least 1 and the parts sum to ``total`` exactly.
    """
    if n <= 0:
        return np.zeros(0, dtype=np.int32)
    if total < n:
        raise ValueError("total must be >= n")
    w = np.exp(rng.normal(0.0, sigma, size=n))
    spare = total - n
    raw = w / w.sum() * spare
    base = np.floor(raw).astype(np.int64)
    rem = spare - int(base.sum())
    order = np.argsort(-(raw - base), kind="stable")
    base[order[:rem]] += 1
    out = base + 1
    assert int(out.sum()) == total
    return out.astype(np.int32)


def _assign_pages(rng: np.random.Generator, num_pool_pages: int, prefix_lens, cur_lens, page_size):
    n_pfx = int((np.asarray(prefix_lens) // page_size).sum())
    n_cur = int(pages_per_len(cur_lens, page_size).sum())
    need = n_pfx + n_cur
    if need > num_pool_pages - 1:
        raise ValueError(f"pool of {num_pool_pages} pages cannot hold {need} pages")
    perm = rng.permutation(np.arange(1, num_pool_pages, dtype=np.int64))
    return perm[:n_pfx].astype(np.int32), perm[n_pfx:need].astype(np.int32)


def round_robin_writers(C: int, cp_size: int) -> np.ndarray:
    """Writer rank of current page i is ``i % cp_size`` (round-robin over pages)."""
    return (np.arange(C, dtype=np.int64) % cp_size).astype(np.int32)


def contiguous_writers(cur_lens, page_size: int, cp_size: int) -> np.ndarray:
    """In-seq contiguous split: each request's current pages are cut into
    cp_size contiguous blocks and block r is written by rank r."""
    out = []
    for n in pages_per_len(cur_lens, page_size).tolist():
        local = np.arange(n, dtype=np.int64)
        out.append((local * cp_size) // max(n, 1))
    return (np.concatenate(out) if out else np.zeros(0, np.int64)).astype(np.int32)


def make_compose_batch(
    name: str,
    seed: int,
    *,
    page_size: int,
    cp_size: int,
    num_pool_pages: int,
    row_bytes: int,
    prefix_lens,
    cur_lens,
    num_layers: int = 1,
    row_kind: str = "bf16",
    writer=None,
    rng: np.random.Generator | None = None,
    prefix_pages=None,
    cur_pages=None,
) -> ComposeBatch:
    """Assemble a batch from explicit lengths; pages come from a seeded permutation."""
    rng = rng if rng is not None else np.random.default_rng(seed)
    prefix_lens = np.asarray(prefix_lens, dtype=np.int32)
    cur_lens = np.asarray(cur_lens, dtype=np.int32)
    if prefix_pages is None or cur_pages is None:
        pp, cpg = _assign_pages(rng, num_pool_pages, prefix_lens, cur_lens, page_size)
        prefix_pages = pp if prefix_pages is None else prefix_pages
        cur_pages = cpg if cur_pages is None else cur_pages
    prefix_pages = np.asarray(prefix_pages, dtype=np.int32)
    cur_pages = np.asarray(cur_pages, dtype=np.int32)
    C = int(cur_pages.shape[0])
    if writer is None:
        writer = round_robin_writers(C, cp_size)
    writer = np.asarray(writer, dtype=np.int32)
    return ComposeBatch(
        name=name,
        seed=seed,
        page_size=page_size,
        cp_size=cp_size,
        num_pool_pages=num_pool_pages,
        row_bytes=row_bytes,
        num_layers=num_layers,
        prefix_lens=prefix_lens,
        cur_lens=cur_lens,
        prefix_pages=prefix_pages,
        cur_pages=cur_pages,
        writer=writer,
        row_kind=row_kind,
    )


def tiny_batch(seed: int = 1001) -> ComposeBatch:
    """Tiny CPU-checkable compose: ps=16, cp=2, B=4, prefix U[0,64] floored to a
    page, current U[1,48], 576-wide bf16 rows, 256-page pool, shuffled pages,
    writers alternating by page."""
    rng = np.random.default_rng(seed)
    ps, B = 16, 4
    pfx = (rng.integers(0, 64 + 1, size=B) // ps) * ps
    cur = rng.integers(1, 48 + 1, size=B)
    return make_compose_batch(
        "tiny", seed, page_size=ps, cp_size=2, num_pool_pages=256,
        row_bytes=MLA_ROW_BYTES, prefix_lens=pfx, cur_lens=cur, rng=rng,
    )


def traced_batch(seed: int = 1002, *, num_layers: int = 1, num_pool_pages: int = 200_000) -> ComposeBatch:
    """Traced prefill shape: ps=64, cp=8, bs=12, 44 600 current tokens split
    lognormally, prefix U[0,16384] floored to a page, MLA 576xbf16 rows,
    randomly permuted pool pages, writers round-robin over pages."""
    rng = np.random.default_rng(seed)
    ps, B = 64, 12
    cur = lognormal_split(rng, 44_600, B)
    pfx = (rng.integers(0, 16384 + 1, size=B) // ps) * ps
    return make_compose_batch(
        "traced", seed, page_size=ps, cp_size=8, num_pool_pages=num_pool_pages,
        row_bytes=MLA_ROW_BYTES, prefix_lens=pfx, cur_lens=cur, rng=rng, num_layers=num_layers,
    )


def traced_78_layer_batch(seed: int = 1002) -> ComposeBatch:
    """The traced batch over 78 layers.  Each layer has its own pool slab of
    4096 pages (8 owners x 512), so the batch's page ids are drawn from
    [1, 4096); every layer indexes its own slab with the same ids."""
    return traced_batch(seed, num_layers=78, num_pool_pages=4096)


def traced_78_token_pages_batch(seed: int = 1006) -> ComposeBatch:
    """The traced batch's lengths over 78 layers with pages of one token
    (page_size = 1, a 1152-byte page per token): 88 832 prefix and 44 600
    current pages per layer.  Each layer has its own pool slab of 2^18 pages
    (8 owners x 32 768); page ids are a seeded permutation inside it and the
    writers go round-robin over pages."""
    tb = traced_batch()
    rng = np.random.default_rng(seed)
    return make_compose_batch(
        "traced_ps1", seed, page_size=1, cp_size=8, num_pool_pages=1 << 18, row_bytes=MLA_ROW_BYTES,
        prefix_lens=tb.prefix_lens, cur_lens=tb.cur_lens, rng=rng, num_layers=78,
    )


def fp8_nsa_batch(seed: int = 1004, *, num_layers: int = 78, num_pool_pages: int = 1 << 20) -> ComposeBatch:
    """FP8 NSA layout: ps=64, cp=8, bs=32, 131 072 current tokens split
    lognormally, prefix U[0,65536] floored to a page, 656-byte rows of random
    bytes, one pool of 2^20 pages shared by all layers."""
    rng = np.random.default_rng(seed)
    ps, B = 64, 32
    cur = lognormal_split(rng, 131_072, B)
    pfx = (rng.integers(0, 65536 + 1, size=B) // ps) * ps
    return make_compose_batch(
        "fp8_nsa", seed, page_size=ps, cp_size=8, num_pool_pages=num_pool_pages,
        row_bytes=NSA_FP8_ROW_BYTES, prefix_lens=pfx, cur_lens=cur, rng=rng,
        num_layers=num_layers, row_kind="bytes",
    )


# ---------------------------------------------------------------------------
# KV bytes
# ---------------------------------------------------------------------------

def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest even) and return the 16-bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = np.isnan(x)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    out = rounded.astype(np.uint16)
    out[nan] = 0x7FC0
    return out


def random_rows(rng: np.random.Generator, n_rows: int, row_bytes: int, kind: str) -> np.ndarray:
    """``n_rows`` KV rows as a [n_rows, row_bytes] uint8 array."""
    if kind == "bf16":
        assert row_bytes % 2 == 0
        vals = rng.standard_normal(size=(n_rows, row_bytes // 2), dtype=np.float32)
        return bf16_bits(vals).view(np.uint8).reshape(n_rows, row_bytes)
    if kind == "bytes":
        return np.frombuffer(rng.bytes(n_rows * row_bytes), dtype=np.uint8).reshape(n_rows, row_bytes).copy()
    raise ValueError(kind)


def host_pool(batch: ComposeBatch, layer: int = 0) -> list[np.ndarray]:
    """Pool slabs of one layer on the host: ``cp`` arrays [slab_pages, ps, R] uint8."""
    rng = np.random.default_rng([batch.seed, 7, layer])
    shape = (batch.slab_pages, batch.page_size, batch.row_bytes)
    slabs = []
    for _ in range(batch.cp_size):
        rows = random_rows(rng, shape[0] * shape[1], shape[2], batch.row_kind)
        slabs.append(rows.reshape(shape))
    return slabs


def host_current_rows(batch: ComposeBatch, layer: int = 0) -> np.ndarray:
    """Current-token KV rows of one layer in batch order: [T, R] uint8."""
    rng = np.random.default_rng([batch.seed, 11, layer])
    return random_rows(rng, batch.T, batch.row_bytes, batch.row_kind)


def token_writer(batch: ComposeBatch) -> np.ndarray:
    """Writer rank of every current token (the writer of the page holding it)."""
    ps = batch.page_size
    out = np.empty(batch.T, dtype=np.int32)
    t = 0
    page = 0
    for n in batch.cur_lens.tolist():
        for k in range(0, n, ps):
            m = min(ps, n - k)
            out[t:t + m] = batch.writer[page]
            t += m
            page += 1
    return out


def split_rows_by_writer(batch: ComposeBatch, rows: np.ndarray) -> list[np.ndarray]:
    """Hand each writer rank the rows of the tokens it computes, in batch order."""
    tw = token_writer(batch)
    return [np.ascontiguousarray(rows[tw == w]) for w in range(batch.cp_size)]


# ---------------------------------------------------------------------------
# Ragged index plan inputs
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class RaggedBatch:
    name: str
    seed: int
    cp_size: int
    chunk: int
    k_align: int
    prefix_lens: np.ndarray  # [B] int32
    q_lens: np.ndarray  # [B] int32

    @property
    def B(self) -> int:
        return int(self.q_lens.shape[0])

    @property
    def num_chunks(self) -> int:
        return int(pages_per_len(self.q_lens, self.chunk).sum())

    split: str = "interleaved"
    topk: int = 2048  # the NSA indexer's selected keys per query (the consumer's index width)

    def cp_index(self, rank: int) -> np.ndarray:
        """Chunk ids owned by ``rank``, ascending, under the batch's split:

        interleaved  global chunk id modulo cp_size (the default);
        contiguous   each request's chunks cut into cp_size contiguous blocks
                     (in-seq split), rank r takes block r of every request;
        zigzag       each request's chunks dealt to 2*cp_size slots, rank r
                     owning slots r and 2*cp_size-1-r (load-balanced causal
                     split).
        """
        if self.split == "interleaved":
            ids = np.arange(self.num_chunks, dtype=np.int64)
            return ids[ids % self.cp_size == rank].astype(np.int32)
        out = []
        first = 0
        for n in pages_per_len(self.q_lens, self.chunk).tolist():
            local = np.arange(n, dtype=np.int64)
            if self.split == "contiguous":
                owner = (local * self.cp_size) // max(n, 1)
                mine = owner == rank
            elif self.split == "zigzag":
                slot = (local * 2 * self.cp_size) // max(n, 1)
                mine = (slot == rank) | (slot == 2 * self.cp_size - 1 - rank)
            else:
                raise ValueError(self.split)
            out.append(first + local[mine])
            first += n
        return (np.concatenate(out) if out else np.zeros(0, np.int64)).astype(np.int32)


def ragged_batch(seed: int = 1005) -> RaggedBatch:
    """Ragged plan config: bs=64, q lens lognormal with total 131 072 (mean 2K),
    prefix U[0,65536], chunk 64, cp=8 interleaved."""
    rng = np.random.default_rng(seed)
    B = 64
    q = lognormal_split(rng, 131_072, B)
    pfx = rng.integers(0, 65536 + 1, size=B).astype(np.int32)
    return RaggedBatch("ragged", seed, cp_size=8, chunk=64, k_align=1, prefix_lens=pfx, q_lens=q)


def ragged_from_compose(batch: ComposeBatch, chunk: int | None = None) -> RaggedBatch:
    """The indexer view of a compose batch: q tokens are the current tokens."""
    return RaggedBatch(
        batch.name + "_ragged", batch.seed, cp_size=batch.cp_size,
        chunk=chunk or batch.page_size, k_align=1,
        prefix_lens=batch.prefix_lens.copy(), q_lens=batch.cur_lens.copy(),
    )


INDEX_K_PLANES = (128, 4)  # NSA indexer key: 128 fp8 bytes, then a 4-byte fp32 scale plane


def index_k_batch(seed: int = 1004, *, num_layers: int = 78, num_pool_pages: int = 1 << 20) -> ComposeBatch:
    """The NSA indexer keys of the fp8 NSA batch (same lengths, pages and
    writers): planar pages of 64 tokens x (128 + 4) bytes = 8448 bytes."""
    b = fp8_nsa_batch(seed, num_layers=num_layers, num_pool_pages=num_pool_pages)
    return dataclasses.replace(b, name="index_k", row_bytes=sum(INDEX_K_PLANES), planes=INDEX_K_PLANES,
                               row_kind="bytes")


def split_planes(rows: np.ndarray, planes) -> list:
    """[n, sum(planes)] rows -> per-plane contiguous [n, w_p] arrays."""
    out, start = [], 0
    for w in planes:
        out.append(np.ascontiguousarray(rows[:, start:start + w]))
        start += w
    return out


CONFIGS = {
    "tiny": tiny_batch,
    "traced": traced_batch,
    "traced_78": traced_78_layer_batch,
    "traced_78_ps1": traced_78_token_pages_batch,
    "fp8_nsa": fp8_nsa_batch,
    "index_k": index_k_batch,
}


def describe(batch: ComposeBatch) -> dict:
    return {
        "B": batch.B,
        "T": batch.T,
        "C": batch.C,
        "prefix_pages": batch.num_prefix_pages,
        "prefix_tokens": int(batch.prefix_lens.sum()),
        "page_size": batch.page_size,
        "cp_size": batch.cp_size,
        "row_bytes": batch.row_bytes,
        "num_pool_pages": batch.num_pool_pages,
        "num_layers": batch.num_layers,
    }


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


__all__ = [
    "ComposeBatch", "RaggedBatch", "MLA_ROW_BYTES", "NSA_FP8_ROW_BYTES", "CONFIGS", "contiguous_writers",
    "tiny_batch", "traced_batch", "traced_78_layer_batch", "fp8_nsa_batch", "ragged_batch",
    "ragged_from_compose", "make_compose_batch", "lognormal_split", "round_robin_writers",
    "random_rows", "host_pool", "host_current_rows", "token_writer", "split_rows_by_writer",
    "bf16_bits", "pages_per_len", "describe", "ceil_div", "index_k_batch", "split_planes", "INDEX_K_PLANES",
]


# ---------------------------------------------------------------------------
# device-side generation (large configs): seeded torch generators on the GPU
# ---------------------------------------------------------------------------

def device_random_rows(n_rows: int, row_bytes: int, kind: str, seed, device="cuda"):
    """[n_rows, row_bytes] uint8 CUDA tensor: bf16 N(0,1) values or uniform bytes."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(int(np.random.SeedSequence(seed).generate_state(1, np.uint64)[0] & 0x7FFFFFFFFFFFFFFF))
    if kind == "bf16":
        x = torch.randn((n_rows, row_bytes // 2), dtype=torch.float32, device=device, generator=g)
        return x.to(torch.bfloat16).view(torch.uint8).reshape(n_rows, row_bytes)
    return torch.randint(0, 256, (n_rows, row_bytes), dtype=torch.uint8, device=device, generator=g)


def device_pool(batch: ComposeBatch, layer: int = 0, device="cuda"):
    """Pool slabs of one layer on the GPU: ``cp`` uint8 tensors [slab_pages, ps, R]."""
    out = []
    for o in range(batch.cp_size):
        rows = device_random_rows(batch.slab_pages * batch.page_size, batch.row_bytes, batch.row_kind,
                                  [batch.seed, 7, layer, o], device)
        out.append(rows.view(batch.slab_pages, batch.page_size, batch.row_bytes))
    return out


def device_current_rows(batch: ComposeBatch, layer: int = 0, device="cuda"):
    """Current-token rows of one layer on the GPU in batch order: [T, R] uint8."""
    return device_random_rows(batch.T, batch.row_bytes, batch.row_kind, [batch.seed, 11, layer], device)


def device_split_rows_by_writer(batch: ComposeBatch, rows):
    """Per-writer compact row buffers (contiguous CUDA tensors), batch order within a writer."""
    import torch

    tw = torch.from_numpy(token_writer(batch)).to(rows.device)
    return [rows[tw == w].contiguous() for w in range(batch.cp_size)]
