"""Shared helpers for the GPU tests: put a synthetic workload into the CUDA
library's paged cache, run one step, and compare with the FP64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import int8_quantized_paged_tokenwise_gb300 as kvq
import oracle
import workloads as W

BS = W.BLOCK_SIZE


def tdtype(dtype: str):
    return torch.bfloat16 if dtype == "bf16" else torch.float16


def to_dev(bits: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(tdtype(dtype))


def bits_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    """16-bit patterns -> float64 (numpy float16 / bf16 as upper float32 half)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == "fp16":
        return b.view(np.float16).astype(np.float64)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of the output dtype at |x| (normal range; subnormal floor)."""
    ax = np.maximum(np.abs(x), 1e-30)
    e = np.floor(np.log2(ax))
    if dtype == "fp16":
        return 2.0 ** np.maximum(e - 10, -24)
    return 2.0 ** np.maximum(e - 7, -133)


ATOL = 2e-3          # max-abs bound for attention outputs
COS_MIN = 0.9999     # cosine similarity bound


def assert_attention_close(gpu_bits: np.ndarray, ref: np.ndarray, dtype: str, what="",
                           v_scale: float = 1.0, atol_extra: float = 0.0):
    """|gpu - oracle| <= 2e-3 * v_scale + half an output ulp elementwise,
    cosine >= 0.9999.

    The half ulp is the rounding of the result to the output dtype, which the
    oracle's unrounded FP64 value does not include; for a BF16 output of
    magnitude ~1 it alone is up to 3.9e-3.  ``v_scale``: the values V were
    multiplied by a power of two v_scale (the workloads' V is N(0,1)-sized);
    attention is linear in V and such a factor leaves every code unchanged
    and multiplies every scale by it, so the absolute bound scales with it.
    ``atol_extra``: a further absolute allowance a caller derives for its own
    arithmetic (the BF16 twin's BF16 softmax weights)."""
    g = bits_f64(gpu_bits, dtype)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - ref)
    tol = ATOL * v_scale + atol_extra + 0.5 * ulp(ref, dtype)
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements out of tolerance, "
                           f"max err {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    gf, rf = g.ravel(), ref.ravel()
    nr = np.linalg.norm(rf) * np.linalg.norm(gf)
    if nr > 0:
        cos = float(gf @ rf / nr)
        assert cos >= COS_MIN, f"{what}: cosine {cos}"
    return float(err.max())


class Case:
    """A workload resident on the GPU: INT8 cache (and optionally the 16-bit
    twin cache), block tables, context lengths and queries."""

    def __init__(self, w: W.Workload, int8=True, kv16=False, device="cuda"):
        self.w = w
        self.device = device
        nb, bt, _ = w.tables()
        self.nb = nb
        self.bt = torch.from_numpy(bt).to(device)
        self.cl = torch.from_numpy(w.context_lens.astype(np.int32)).to(device)
        self.q = to_dev(w.q_all(), w.dtype, device)
        self.int8 = kvq.alloc_int8_cache(nb, w.num_kv_heads, w.head_dim, device) if int8 else None
        self.kv16 = (kvq.alloc_kv16_cache(nb, w.num_kv_heads, w.head_dim, tdtype(w.dtype), device)
                     if kv16 else None)

    def _write(self, k_bits, v_bits, slots):
        if len(slots) == 0:
            return
        k = to_dev(k_bits, self.w.dtype, self.device)
        v = to_dev(v_bits, self.w.dtype, self.device)
        s = torch.from_numpy(np.ascontiguousarray(slots, dtype=np.int64)).to(self.device)
        if self.int8 is not None:
            kvq.kvq_quantize_append(k, v, s, *self.int8)
        if self.kv16 is not None:
            kvq.kvq_cache_append_kv16(k, v, s, *self.kv16)

    def write_prefix(self):
        """Setup: every token already in the cache before the step."""
        w = self.w
        for b in range(w.num_seqs):
            k, v = w.seq_kv(b)
            n = int(w.prefix_lens[b])
            self._write(k[:n], v[:n], w.slots(b, 0, n))

    def step_inputs(self):
        """(k, v, slots) of one step's quantize-append: the appended token of
        every sequence, then the prefill chunk."""
        w = self.w
        ks, vs, ss = [], [], []
        if w.append:
            for b in range(w.num_seqs):
                k, v = w.seq_kv(b)
                L = int(w.context_lens[b])
                ks.append(k[L - 1:L]); vs.append(v[L - 1:L]); ss.append(w.slots(b, L - 1, L))
        if w.prefill_tokens:
            pk, pv = w.prefill_kv()
            ks.append(pk); vs.append(pv); ss.append(w.prefill_slots())
        if not ks:
            e = np.zeros((0, w.num_kv_heads, w.head_dim), np.uint16)
            return e, e, np.zeros(0, np.int64)
        return np.concatenate(ks), np.concatenate(vs), np.concatenate(ss)

    def write_step(self):
        k, v, s = self.step_inputs()
        self._write(k, v, s)

    def decode(self, partition_pages=0, kv16=False):
        w = self.w
        if kv16:
            return kvq.kvq_paged_decode_kv16(self.q, *self.kv16, self.bt, self.cl,
                                             w.max_context_len, w.sm_scale,
                                             partition_pages=partition_pages)
        return kvq.kvq_paged_decode(self.q, *self.int8, self.bt, self.cl, w.max_context_len,
                                    w.sm_scale, partition_pages=partition_pages)

    def gather_seq(self, b: int):
        """INT8 codes/scales of sequence b read back through its block table:
        (k codes [L,Hkv,D], v codes, k scale bits [L,Hkv], v scale bits)."""
        L = int(self.w.context_lens[b])
        t = torch.arange(L, device=self.device)
        blk = self.bt[b, t // BS].long()
        off = t % BS
        kc, vc, ks, vs = self.int8
        return (kc[blk, :, off].cpu().numpy(), vc[blk, :, off].cpu().numpy(),
                ks[blk, :, off].cpu().numpy().view(np.uint16),
                vs[blk, :, off].cpu().numpy().view(np.uint16))


def out_bits(out: torch.Tensor) -> np.ndarray:
    return out.cpu().view(torch.int16).numpy().view(np.uint16)
