"""Seeded synthetic inputs for the INT8 paged KV-cache path.

This module is shared by the tests, the benchmark, the smoke check and the CPU
oracle's callers.  It holds input recipes only -- shapes, distributions, block
tables and slot mappings -- and none of the quantization or attention
arithmetic.  Values are produced as 16-bit patterns (numpy ``uint16``) so that
exactly the same bits feed the oracle and the CUDA library.

Every per-sequence array is drawn from its own counter-style seed
``(workload seed, workload id, sequence, stream)``, so any single sequence can
be regenerated on its own (the oracle checks sampled sequences of the large
workloads without generating the rest).

Workloads (all block_size 16, sm_scale = 1/sqrt(head_dim)):

* ``tiny``      2 seqs, contexts 17 and 40, 4 query / 2 KV heads, d 64, fp16,
                Q,K,V ~ N(0,1); all tokens quantize-appended, then one decode.
* ``canonical`` 32 seqs, contexts ~ U[512, 2048] plus one appended token,
                32 / 8 heads, d 128, bf16, N(0,1); block pool twice the need.
* ``long``      4 seqs x 32768, 32 / 8 heads, d 128, bf16; K ~ N(0,1) with 4
                fixed outlier channels per KV head scaled x20; V ~ N(0,1).
* ``mha``       64 seqs x 4096, 32 / 32 heads, d 128, fp16, K,V ~ N(0, 0.5^2),
                1 % of token positions all-zero (K and V, every head).
* ``serving``   256 seqs, contexts lognormal(median 1024, sigma 1) clipped to
                [16, 16384] plus one appended token, 64 / 8 heads, d 128, bf16,
                fragmented (shuffled) block pool, plus one 8192-token prefill
                chunk written per step into a separate sequence's pages.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 16
_IDS = {"tiny": 0, "canonical": 1, "long": 2, "mha": 3, "serving": 4, "custom": 9}
_STREAM = {"k": 1, "v": 2, "q": 3, "newk": 4, "newv": 5, "pk": 6, "pv": 7, "zero": 8}


def _rng(seed: int, wid: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, wid, *key])))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even float32 -> bfloat16 bit patterns (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 samples -> 16-bit patterns of the workload dtype (RNE)."""
    if dtype == "fp16":
        return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    raise ValueError(dtype)


@dataclass
class Workload:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    dtype: str
    context_lens: np.ndarray          # tokens attended at the decode step, [B] int32
    append: bool                      # a step appends one token per sequence first
    prefill_tokens: int = 0           # tokens of a separate prefill chunk per step
    k_std: float = 1.0
    v_std: float = 1.0
    q_std: float = 1.0
    outlier_channels: int = 0         # per KV head, K only
    outlier_gain: float = 1.0
    zero_token_frac: float = 0.0
    pool_factor: int = 2
    seed: int = 0
    block_size: int = BLOCK_SIZE
    _outliers: np.ndarray | None = field(default=None, repr=False)
    _tables: tuple | None = field(default=None, repr=False)

    # ------------------------------------------------------------ shapes ---
    @property
    def wid(self) -> int:
        return _IDS.get(self.name, _IDS["custom"])

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def prefix_lens(self) -> np.ndarray:
        """Tokens already in the cache before a step's append."""
        return self.context_lens - (1 if self.append else 0)

    def pages(self, n: int) -> int:
        return (int(n) + self.block_size - 1) // self.block_size

    # ------------------------------------------------------- block tables ---
    def tables(self):
        """(num_blocks, block_tables [B, max_blocks] int32, prefill_blocks [n] int32).

        Pages for every sequence (and the prefill chunk) are taken in order from
        a random permutation of a pool ``pool_factor`` times the required size,
        so logically adjacent pages are physically scattered."""
        if self._tables is None:
            need = [self.pages(L) for L in self.context_lens]
            pf = self.pages(self.prefill_tokens)
            total = sum(need) + pf
            nb = max(1, self.pool_factor * total)
            perm = _rng(self.seed, self.wid, 1000).permutation(nb).astype(np.int32)
            maxb = max(need) if need else 0
            bt = np.full((self.num_seqs, max(maxb, 1)), -1, dtype=np.int32)
            pos = 0
            for b, n in enumerate(need):
                bt[b, :n] = perm[pos:pos + n]
                pos += n
            pre = perm[pos:pos + pf].copy()
            self._tables = (nb, bt, pre)
        return self._tables

    @property
    def num_blocks(self) -> int:
        return self.tables()[0]

    @property
    def block_tables(self) -> np.ndarray:
        return self.tables()[1]

    def slots(self, b: int, t0: int, t1: int) -> np.ndarray:
        """Slot ids (block * bs + offset) of tokens [t0, t1) of sequence b."""
        t = np.arange(t0, t1, dtype=np.int64)
        bt = self.block_tables[b]
        return bt[t // self.block_size].astype(np.int64) * self.block_size + t % self.block_size

    def prefill_slots(self) -> np.ndarray:
        t = np.arange(self.prefill_tokens, dtype=np.int64)
        pre = self.tables()[2]
        return pre[t // self.block_size].astype(np.int64) * self.block_size + t % self.block_size

    # ------------------------------------------------------------- values ---
    def _outlier_idx(self) -> np.ndarray:
        if self._outliers is None:
            r = _rng(self.seed, self.wid, 2000)
            self._outliers = np.stack([r.choice(self.head_dim, self.outlier_channels, replace=False)
                                       for _ in range(self.num_kv_heads)]) \
                if self.outlier_channels else np.zeros((self.num_kv_heads, 0), dtype=np.int64)
        return self._outliers

    def _draw(self, n: int, std: float, *key: int) -> np.ndarray:
        r = _rng(self.seed, self.wid, *key)
        x = r.standard_normal((n, self.num_kv_heads, self.head_dim), dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        return x

    def seq_kv(self, b: int):
        """All tokens of sequence b as written to the cache: (k, v) bits
        [context_len, Hkv, D].  With ``append`` the last token is the one the
        decode step appends."""
        L = int(self.context_lens[b])
        k = self._draw(L, self.k_std, _STREAM["k"], b)
        v = self._draw(L, self.v_std, _STREAM["v"], b)
        if self.outlier_channels:
            idx = self._outlier_idx()
            for j in range(self.num_kv_heads):
                k[:, j, idx[j]] *= np.float32(self.outlier_gain)
        if self.zero_token_frac > 0.0 and L > 0:
            nz = int(math.floor(self.zero_token_frac * L))
            if nz:
                zr = _rng(self.seed, self.wid, _STREAM["zero"], b)
                pos = zr.choice(L, nz, replace=False)
                k[pos] = 0.0
                v[pos] = 0.0
        return to_bits(k, self.dtype), to_bits(v, self.dtype)

    def seq_q(self, b: int) -> np.ndarray:
        r = _rng(self.seed, self.wid, _STREAM["q"], b)
        x = r.standard_normal((self.num_q_heads, self.head_dim), dtype=np.float32)
        if self.q_std != 1.0:
            x *= np.float32(self.q_std)
        return to_bits(x, self.dtype)

    def q_all(self) -> np.ndarray:
        if self.num_seqs == 0:
            return np.zeros((0, self.num_q_heads, self.head_dim), dtype=np.uint16)
        return np.stack([self.seq_q(b) for b in range(self.num_seqs)])

    def prefill_kv(self):
        n = self.prefill_tokens
        k = self._draw(n, self.k_std, _STREAM["pk"])
        v = self._draw(n, self.v_std, _STREAM["pv"])
        return to_bits(k, self.dtype), to_bits(v, self.dtype)

    # ---------------------------------------------- device-side draws ---
    def _torch_draw(self, n: int, std: float, device, *key: int):
        import torch
        state = np.random.SeedSequence([self.seed, self.wid, *key]).generate_state(2, np.uint32)
        g = torch.Generator(device=device)
        g.manual_seed((int(state[0]) << 31) ^ int(state[1]))
        x = torch.randn((n, self.num_kv_heads, self.head_dim), generator=g, device=device,
                        dtype=torch.float32)
        if std != 1.0:
            x *= std
        return x

    def _torch_dtype(self):
        import torch
        return torch.bfloat16 if self.dtype == "bf16" else torch.float16

    def seq_kv_device(self, b: int, device):
        """seq_kv's recipe drawn on the device with torch's generator: the same
        distribution, outlier channels and all-zero token positions, another
        stream of N(0, 1) numbers.  Returns (k, v) tensors [L, Hkv, D] of the
        workload dtype (RNE from float32).  For timing runs, where numpy draws
        of the large workloads would take a minute."""
        L = int(self.context_lens[b])
        k = self._torch_draw(L, self.k_std, device, _STREAM["k"], b)
        v = self._torch_draw(L, self.v_std, device, _STREAM["v"], b)
        if self.outlier_channels:
            idx = self._outlier_idx()
            for j in range(self.num_kv_heads):
                k[:, j, list(idx[j])] *= float(self.outlier_gain)
        if self.zero_token_frac > 0.0 and L > 0:
            nz = int(math.floor(self.zero_token_frac * L))
            if nz:
                zr = _rng(self.seed, self.wid, _STREAM["zero"], b)
                pos = list(zr.choice(L, nz, replace=False))
                k[pos] = 0.0
                v[pos] = 0.0
        return k.to(self._torch_dtype()), v.to(self._torch_dtype())

    def prefill_kv_device(self, device):
        n = self.prefill_tokens
        k = self._torch_draw(n, self.k_std, device, _STREAM["pk"])
        v = self._torch_draw(n, self.v_std, device, _STREAM["pv"])
        return k.to(self._torch_dtype()), v.to(self._torch_dtype())

    # ---------------------------------------------------- byte accounting ---
    def decode_bytes_int8_seq(self, L: int) -> int:
        """decode_bytes_int8's share of one sequence with context L."""
        return (int(L) * self.num_kv_heads * (2 * self.head_dim + 4) + self.pages(L) * 4 +
                2 * self.num_q_heads * self.head_dim * 2 + 4)

    def decode_bytes_int8(self) -> int:
        """Algorithmic HBM bytes of one INT8 decode: K/V payload + scales of the
        attended tokens, the block-table entries read, q and out."""
        L = self.context_lens.astype(np.int64)
        kv = int(L.sum()) * self.num_kv_heads * (2 * self.head_dim + 4)
        bt = sum(self.pages(x) for x in L) * 4
        qo = 2 * self.num_seqs * self.num_q_heads * self.head_dim * 2
        return kv + bt + qo + 4 * self.num_seqs

    def decode_bytes_kv16(self) -> int:
        L = self.context_lens.astype(np.int64)
        kv = int(L.sum()) * self.num_kv_heads * 4 * self.head_dim
        bt = sum(self.pages(x) for x in L) * 4
        qo = 2 * self.num_seqs * self.num_q_heads * self.head_dim * 2
        return kv + bt + qo + 4 * self.num_seqs

    def append_tokens(self) -> int:
        return (self.num_seqs if self.append else 0) + self.prefill_tokens

    def append_bytes_int8(self) -> int:
        """Read 16-bit K and V rows, write codes + FP16 scales, read slots."""
        n = self.append_tokens() * self.num_kv_heads
        return n * 2 * (2 * self.head_dim) + n * 2 * (self.head_dim + 2) + self.append_tokens() * 8

    def append_bytes_kv16(self) -> int:
        n = self.append_tokens() * self.num_kv_heads
        return n * 2 * (2 * self.head_dim) * 2 + self.append_tokens() * 8


def first_seqs(w: Workload, n: int) -> Workload:
    """The workload restricted to its first n sequences (same values for
    those sequences; block tables drawn afresh for the smaller pool)."""
    return Workload(w.name, n, w.num_q_heads, w.num_kv_heads, w.head_dim, w.dtype,
                    w.context_lens[:n].copy(), w.append, w.prefill_tokens, w.k_std, w.v_std,
                    w.q_std, w.outlier_channels, w.outlier_gain, w.zero_token_frac,
                    w.pool_factor, w.seed, w.block_size)


def make(name: str, seed: int = 0) -> Workload:
    """The five named workloads."""
    wid = _IDS[name]
    if name == "tiny":
        return Workload("tiny", 2, 4, 2, 64, "fp16", np.array([17, 40], dtype=np.int32),
                        append=False, seed=seed)
    if name == "canonical":
        L = _rng(seed, wid, 10).integers(512, 2048, size=32, endpoint=True).astype(np.int32)
        return Workload("canonical", 32, 32, 8, 128, "bf16", L + 1, append=True, seed=seed)
    if name == "long":
        return Workload("long", 4, 32, 8, 128, "bf16", np.full(4, 32768, dtype=np.int32),
                        append=False, outlier_channels=4, outlier_gain=20.0, seed=seed)
    if name == "mha":
        return Workload("mha", 64, 32, 32, 128, "fp16", np.full(64, 4096, dtype=np.int32),
                        append=False, k_std=0.5, v_std=0.5, zero_token_frac=0.01, seed=seed)
    if name == "serving":
        r = _rng(seed, wid, 10)
        L = np.exp(math.log(1024.0) + 1.0 * r.standard_normal(256))
        L = np.clip(np.rint(L), 16, 16384).astype(np.int32)
        return Workload("serving", 256, 64, 8, 128, "bf16", L + 1, append=True,
                        prefill_tokens=8192, seed=seed)
    raise KeyError(name)


def custom(num_seqs, num_q_heads, num_kv_heads, head_dim, dtype, context_lens, seed=0,
           append=False, pool_factor=2, **kw) -> Workload:
    """A free-form workload (edge cases, sweeps) with N(0,1) values."""
    return Workload("custom", num_seqs, num_q_heads, num_kv_heads, head_dim, dtype,
                    np.asarray(context_lens, dtype=np.int32), append=append,
                    pool_factor=pool_factor, seed=seed, **kw)


NAMES = ("tiny", "canonical", "long", "mha", "serving")
