"""Synthetic decode traces shaped like the PersistentKV evaluation workloads.

Source: "PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM Serving on Commodity GPUs" (arXiv
2606.26666). The abstract fixes the shapes (FP16, page size 16, Hq=32, Hkv=8, d=128) and names the trace families
(B1 bucketed long context; B8 bimodal, uniform and Zipf-like; the B4 bimodal boundary case); the gist.science
technical summary, "Evaluatieprotocol", says the traces are synthetic and built to isolate context length, active
batch size and length raggedness. The pages give no distribution parameters; the ones below are plain readings:
bimodal rows are half short (U[256, 1024]) then half long (U[16384, 32768]); Zipf-like lengths are 256 * k with k
drawn from Zipf(1.1) truncated to 1..128; values are fp16 N(0, 1) through a 16-bit quantile table.

Everything is seeded. Values are drawn with numpy's PCG64 through ``SeedSequence([seed, stream...])`` so the same
seed gives the same trace on any machine. Nothing here computes attention.
"""

from __future__ import annotations

import math
import mmap
from dataclasses import dataclass, field

import numpy as np

HQ, HKV, D, PS = 32, 8, 128, 16

# stream ids for SeedSequence, so lengths, permutations, K, V and q never share random numbers
_S_LEN, _S_PERM, _S_K, _S_V, _S_Q = 1, 2, 3, 4, 5

_NORMAL_TABLE: np.ndarray | None = None


def rng_for(seed: int, *stream: int) -> np.random.Generator:
    """A PCG64 generator for (seed, stream...)."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), *[int(s) for s in stream]])))


def _normal_table() -> np.ndarray:
    # fp16 N(0,1) quantiles at the midpoints of 65536 equal-probability bins: a 16-bit index drawn uniformly maps
    # to a standard-normal value, rounded to fp16. It is much faster than Box-Muller for the GB-sized pools.
    global _NORMAL_TABLE
    if _NORMAL_TABLE is None:
        from scipy.special import ndtri

        _NORMAL_TABLE = ndtri((np.arange(65536, dtype=np.float64) + 0.5) / 65536.0).astype(np.float16)
    return _NORMAL_TABLE


def normal_fp16(rng: np.random.Generator, shape) -> np.ndarray:
    """fp16 values ~ N(0,1) (16-bit quantile resolution, tails at about +-4.3)."""
    n = int(np.prod(shape, dtype=np.int64))
    idx = np.frombuffer(rng.bytes(2 * n), dtype=np.uint16)
    return _normal_table()[idx].reshape(shape)


def lazy_zeros(shape, dtype) -> np.ndarray:
    """A zero-filled array whose memory is committed only where written (anonymous mmap, no huge pages), so a
    GB-sized page pool with a few thousand pages filled costs only those pages."""
    nbytes = int(np.prod(shape, dtype=np.int64)) * np.dtype(dtype).itemsize
    if nbytes < (1 << 22):
        return np.zeros(shape, dtype=dtype)
    buf = mmap.mmap(-1, nbytes)
    if hasattr(mmap, "MADV_NOHUGEPAGE"):
        try:
            buf.madvise(mmap.MADV_NOHUGEPAGE)
        except OSError:
            pass
    return np.frombuffer(buf, dtype=dtype).reshape(shape)


def zipf_lengths(rng: np.random.Generator, n: int, s: float = 1.1, kmax: int = 128, unit: int = 256) -> np.ndarray:
    """L = unit*k with k ~ Zipf(s) truncated to 1..kmax (renormalised pmf ~ k^-s, sampled by inverse CDF)."""
    k = np.arange(1, kmax + 1, dtype=np.float64)
    pmf = k ** (-s)
    cdf = np.cumsum(pmf / pmf.sum())
    u = rng.random(n)
    kk = np.searchsorted(cdf, u, side="right") + 1
    kk = np.minimum(kk, kmax)
    return (unit * kk).astype(np.int64)


@dataclass(frozen=True)
class TraceConfig:
    name: str
    batch: int
    steps: int
    pool_pages: int | None  # None: sized from the trace (stress)
    splits: int | None = None  # fixed split count, where the workload states one
    description: str = ""


CONFIGS: dict[str, TraceConfig] = {
    "tiny": TraceConfig("tiny", 1, 1, 64, splits=4,
                        description="B=1, L=512 (32 pages) in a 64-page pool, split count 4"),
    "b1_bucketed": TraceConfig("b1_bucketed", 1, 64, 1 << 16,
                               description="B=1, start length from {4096, 8192, 16384, 32768}, 64 steps"),
    "b8_bimodal": TraceConfig("b8_bimodal", 8, 64, 1 << 16,
                              description="rows 0-3 ~U[256,1024], rows 4-7 ~U[16384,32768], 64 steps"),
    "b8_uniform": TraceConfig("b8_uniform", 8, 64, 1 << 16, description="8 rows ~U[1024,32768], 64 steps"),
    "b8_zipf": TraceConfig("b8_zipf", 8, 64, 1 << 16,
                           description="8 rows, L=256*k, k ~ Zipf(1.1) truncated to 1..128, 64 steps"),
    "b4_bimodal": TraceConfig("b4_bimodal", 4, 64, 1 << 16,
                              description="rows 0-1 ~U[256,1024], rows 2-3 ~U[16384,32768], 64 steps"),
    "stress": TraceConfig("stress", 64, 4, None,
                          description="B=64, L=round(exp(U[ln 512, ln 131072])), pool min(2^20, ceil(1.25*pages))"),
}


def start_lengths(name: str, seed: int) -> np.ndarray:
    """Context length of every row at step 0 (the token decoded at step 0 is included)."""
    r = rng_for(seed, _S_LEN)
    if name == "tiny":
        return np.array([512], dtype=np.int64)
    if name == "b1_bucketed":
        return np.array([r.choice([4096, 8192, 16384, 32768])], dtype=np.int64)
    if name in ("b8_bimodal", "b4_bimodal"):
        half = 4 if name == "b8_bimodal" else 2
        short = r.integers(256, 1024, size=half, endpoint=True)
        long_ = r.integers(16384, 32768, size=half, endpoint=True)
        return np.concatenate([short, long_]).astype(np.int64)
    if name == "b8_uniform":
        return r.integers(1024, 32768, size=8, endpoint=True).astype(np.int64)
    if name == "b8_zipf":
        return zipf_lengths(r, 8)
    if name == "stress":
        u = r.uniform(math.log(512.0), math.log(131072.0), size=64)
        return np.rint(np.exp(u)).astype(np.int64)
    raise KeyError(name)


@dataclass
class Trace:
    """One seeded decode trace: B rows whose lengths grow by one token per step over a shuffled page pool.

    Step t (0-based) attends over ``seq_lens(t) = start + t`` tokens per row: the harness appends the step's own
    token before the step runs. Pages are taken from a seeded permutation of the pool: first the start pages of
    rows 0..B-1 in order, then, at every step where a row's new token opens a page ((L-1) % 16 == 0), the next
    permutation entry.
    """

    name: str
    seed: int
    batch: int
    steps: int
    num_pages: int
    start: np.ndarray  # int64 [B]
    table: np.ndarray  # int32 [B, max_pages] physical page of each logical page at the last step
    used_pages: np.ndarray  # int64 [n_used] physical ids in allocation order
    page_row: np.ndarray  # int64 [n_used] owning row of each used page
    page_logical: np.ndarray  # int64 [n_used] logical index of each used page within its row
    hq: int = HQ
    hkv: int = HKV
    d: int = D
    ps: int = PS
    _k: np.ndarray | None = field(default=None, repr=False)
    _v: np.ndarray | None = field(default=None, repr=False)

    # ---- lengths and tables -----------------------------------------------------------------------------------
    @property
    def max_pages(self) -> int:
        return int(self.table.shape[1])

    def seq_lens(self, t: int) -> np.ndarray:
        return (self.start + t).astype(np.int32)

    def pages(self, t: int) -> np.ndarray:
        return (self.seq_lens(t).astype(np.int64) + self.ps - 1) // self.ps

    def block_table(self, t: int) -> np.ndarray:
        """int32 [B, max_pages]; entries past a row's last page at step t are -1."""
        p = self.pages(t)
        cols = np.arange(self.max_pages)[None, :]
        return np.where(cols < p[:, None], self.table, -1).astype(np.int32)

    def q(self, t: int) -> np.ndarray:
        return normal_fp16(rng_for(self.seed, _S_Q, t), (self.batch, self.hq, self.d))

    # ---- page contents ----------------------------------------------------------------------------------------
    def _contents(self):
        if self._k is None:
            shape = (len(self.used_pages), self.ps, self.hkv, self.d)
            self._k = normal_fp16(rng_for(self.seed, _S_K), shape)
            self._v = normal_fp16(rng_for(self.seed, _S_V), shape)
        return self._k, self._v

    @property
    def k_pages(self) -> np.ndarray:
        return self._contents()[0]

    @property
    def v_pages(self) -> np.ndarray:
        return self._contents()[1]

    def valid_slots(self, t: int) -> np.ndarray:
        """Per used page, how many of its slots hold tokens at step t (0..page_size)."""
        lens = self.seq_lens(t).astype(np.int64)[self.page_row]
        return np.clip(lens - self.page_logical * self.ps, 0, self.ps)

    def host_pools(self) -> tuple[np.ndarray, np.ndarray]:
        """Full-size fp16 pools [num_pages, ps, Hkv, d] with every used page filled (unused pages are zero).

        The arrays are allocated zeroed, so the untouched part of a large pool is not committed host memory.
        """
        k, v = self._contents()
        shape = (self.num_pages, self.ps, self.hkv, self.d)
        kp = lazy_zeros(shape, np.float16)
        vp = lazy_zeros(shape, np.float16)
        kp[self.used_pages] = k
        vp[self.used_pages] = v
        return kp, vp


def make_trace(name: str, seed: int, steps: int | None = None, pool_pages: int | None = None) -> Trace:
    cfg = CONFIGS[name]
    steps = cfg.steps if steps is None else int(steps)
    start = start_lengths(name, seed)
    batch = len(start)
    final = start + (steps - 1)
    final_pages = (final + PS - 1) // PS
    total_pages = int(final_pages.sum())
    if pool_pages is None:
        pool_pages = cfg.pool_pages
    if pool_pages is None:
        pool_pages = min(1 << 20, int(math.ceil(1.25 * total_pages)))
    if total_pages > pool_pages:
        raise ValueError(f"{name}: trace needs {total_pages} pages, pool has {pool_pages}")

    perm = rng_for(seed, _S_PERM).permutation(pool_pages)
    max_pages = int(final_pages.max())
    table = np.full((batch, max_pages), -1, dtype=np.int32)
    used, rows, logical = [], [], []
    nxt = 0

    def take(b: int, p: int):
        nonlocal nxt
        phys = int(perm[nxt])
        nxt += 1
        table[b, p] = phys
        used.append(phys)
        rows.append(b)
        logical.append(p)

    for b in range(batch):
        for p in range(int((start[b] + PS - 1) // PS)):
            take(b, p)
    lens = start.copy()
    for _t in range(1, steps):
        for b in range(batch):
            lens[b] += 1
            if (lens[b] - 1) % PS == 0:
                take(b, int((lens[b] - 1) // PS))

    return Trace(name=name, seed=int(seed), batch=batch, steps=steps, num_pages=int(pool_pages), start=start,
                 table=table, used_pages=np.array(used, dtype=np.int64), page_row=np.array(rows, dtype=np.int64),
                 page_logical=np.array(logical, dtype=np.int64))
