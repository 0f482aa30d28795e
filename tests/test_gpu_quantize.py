"""Quantize-append on the GPU is bit-exact against the FP64 oracle (codes and
FP16 scale bits), on every workload and on adversarial rows."""
import numpy as np
import pytest
import torch

import int8_quantized_paged_tokenwise_gb300 as kvq
import oracle
import workloads as W
from _harness import Case, to_dev

pytestmark = pytest.mark.gpu


def _check_seq(case: Case, b: int):
    w = case.w
    k, v = w.seq_kv(b)
    gk, gv, gks, gvs = case.gather_seq(b)
    qk, sk = oracle.quantize_rows(k, w.dtype)
    qv, sv = oracle.quantize_rows(v, w.dtype)
    assert np.array_equal(gks, sk), f"seq {b}: K scales differ"
    assert np.array_equal(gvs, sv), f"seq {b}: V scales differ"
    assert np.array_equal(gk, qk), f"seq {b}: K codes differ"
    assert np.array_equal(gv, qv), f"seq {b}: V codes differ"


def test_quantize_bit_exact_tiny():
    case = Case(W.make("tiny"))
    case.write_prefix()
    case.write_step()
    for b in range(case.w.num_seqs):
        _check_seq(case, b)
    assert kvq.kvq_get_error() == (0, 0)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["canonical", "long", "mha", "serving"])
def test_quantize_bit_exact_full_workload(name):
    """Every token of the full workload, including one step's append and (for
    the serving mix) the 8192-token prefill chunk."""
    w = W.make(name)
    case = Case(w)
    case.write_prefix()
    case.write_step()
    torch.cuda.synchronize()
    for b in range(w.num_seqs):
        _check_seq(case, b)
    if w.prefill_tokens:
        pk, pv = w.prefill_kv()
        slots = torch.from_numpy(w.prefill_slots()).cuda()
        kc, vc, ks, vs = case.int8
        blk, off = slots // 16, slots % 16
        qk, sk = oracle.quantize_rows(pk, w.dtype)
        qv, sv = oracle.quantize_rows(pv, w.dtype)
        assert np.array_equal(kc[blk, :, off].cpu().numpy(), qk)
        assert np.array_equal(vc[blk, :, off].cpu().numpy(), qv)
        assert np.array_equal(ks[blk, :, off].cpu().numpy().view(np.uint16), sk)
        assert np.array_equal(vs[blk, :, off].cpu().numpy().view(np.uint16), sv)
    # properties over the whole cache
    kc, vc, _, _ = case.int8
    assert not bool((kc == -128).any()) and not bool((vc == -128).any())
    assert kvq.kvq_get_error() == (0, 0)


def _adversarial_rows(dtype: str, D: int) -> np.ndarray:
    r = np.random.default_rng(5)
    rows = []
    if dtype == "fp16":
        # exact ties x = (k + 1/2) * s for s = 1.0 (a row with absmax 127)
        t = np.arange(D, dtype=np.float64) % 127 - 63 + 0.5
        t[0] = 127.0
        rows.append(t.astype(np.float16).view(np.uint16))
        # subnormal scales: absmax below 127 * 2^-14
        rows.append((r.standard_normal(D) * 1e-4).astype(np.float16).view(np.uint16))
        rows.append((r.standard_normal(D) * 3e-7).astype(np.float16).view(np.uint16))
        # +-max fp16
        m = np.full(D, 65504.0); m[1::2] = -65504.0
        rows.append(m.astype(np.float16).view(np.uint16))
        # single nonzero element, smallest subnormal
        s = np.zeros(D, np.uint16); s[3] = 1
        rows.append(s)
    else:
        rows.append(W.f32_to_bf16_bits((r.standard_normal(D) * 1e-30).astype(np.float32)))
        tiny = np.zeros(D, np.uint16); tiny[5] = 0x0001; tiny[9] = 0x8003   # bf16 subnormals
        rows.append(tiny)
        big = (r.standard_normal(D) * 1e7).astype(np.float32)              # saturated scale
        rows.append(W.f32_to_bf16_bits(big))
        t = (np.arange(D) % 255 - 127).astype(np.float32) * np.float32(2.0 ** -3)
        rows.append(W.f32_to_bf16_bits(t))
    rows.append(np.zeros(D, np.uint16))                                     # all-zero token
    neg0 = np.full(D, 0x8000, np.uint16)                                    # all -0.0
    rows.append(neg0)
    # random rows at many magnitudes
    for e in range(-12, 5, 2):
        x = (r.standard_normal(D) * 10.0 ** e).astype(np.float32)
        rows.append(W.to_bits(x, dtype))
    return np.stack(rows)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
def test_quantize_adversarial_rows(dtype, D):
    rows = _adversarial_rows(dtype, D)
    T = rows.shape[0]
    Hkv = 1
    k = rows[:, None, :]
    v = rows[::-1].copy()[:, None, :]
    nb = (T + 15) // 16 + 3
    kc, vc, ks, vs = kvq.alloc_int8_cache(nb, Hkv, D)
    kc.fill_(7); vc.fill_(7); ks.fill_(7); vs.fill_(7)
    perm = np.random.default_rng(1).permutation(nb * 16)[:T].astype(np.int64)
    perm[2] = -1                                                          # skipped token
    kvq.kvq_quantize_append(to_dev(k, dtype), to_dev(v, dtype), torch.from_numpy(perm).cuda(),
                            kc, vc, ks, vs)
    kcn, vcn = kc.cpu().numpy(), vc.cpu().numpy()
    ksn, vsn = ks.cpu().numpy().view(np.uint16), vs.cpu().numpy().view(np.uint16)
    qk, sk = oracle.quantize_rows(k, dtype)
    qv, sv = oracle.quantize_rows(v, dtype)
    for t in range(T):
        if perm[t] < 0:
            continue
        blk, off = perm[t] // 16, perm[t] % 16
        assert np.array_equal(kcn[blk, 0, off], qk[t, 0]) and ksn[blk, 0, off] == sk[t, 0], t
        assert np.array_equal(vcn[blk, 0, off], qv[t, 0]) and vsn[blk, 0, off] == sv[t, 0], t
    # untouched slots keep their bytes (nothing written for the skipped token)
    written = set(int(s) for s in perm if s >= 0)
    for s in range(nb * 16):
        if s not in written:
            assert np.all(kcn[s // 16, 0, s % 16] == 7) and ksn[s // 16, 0, s % 16] == 7
    assert kvq.kvq_get_error() == (0, 0)


def test_quantize_out_of_range_slot_sets_error_bit():
    D, Hkv = 64, 2
    kc, vc, ks, vs = kvq.alloc_int8_cache(2, Hkv, D)
    k = torch.randn(3, Hkv, D, device="cuda", dtype=torch.float16)
    slots = torch.tensor([0, 2 * 16, 5], dtype=torch.int64, device="cuda")   # middle one bad
    kvq.kvq_quantize_append(k, k, slots, kc, vc, ks, vs)
    st, flags = kvq.kvq_get_error()
    assert st == 5 and flags & kvq.DEVERR_SLOT
    assert kvq.kvq_get_error() == (0, 0)                                    # cleared
    assert bool((ks[0, :, 0] != 0).all()) and bool((ks[0, :, 5] != 0).all())


def test_quantize_host_validation():
    D, Hkv = 64, 2
    kc, vc, ks, vs = kvq.alloc_int8_cache(2, Hkv, D)
    k = torch.randn(3, Hkv, D, device="cuda", dtype=torch.float16)
    slots = torch.zeros(3, dtype=torch.int64, device="cuda")
    L = kvq.load()
    import ctypes
    st = L.kvq_quantize_append(ctypes.c_void_p(k.data_ptr()), None, Hkv * D, Hkv * D, 3, Hkv, D,
                               0, ctypes.c_void_p(slots.data_ptr()),
                               ctypes.c_void_p(kc.data_ptr()), ctypes.c_void_p(vc.data_ptr()),
                               ctypes.c_void_p(ks.data_ptr()), ctypes.c_void_p(vs.data_ptr()),
                               2, 16, None)
    assert st == 1                                                          # NULL v
    st = L.kvq_quantize_append(ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                               Hkv * D, Hkv * D, 3, Hkv, 96, 0, ctypes.c_void_p(slots.data_ptr()),
                               ctypes.c_void_p(kc.data_ptr()), ctypes.c_void_p(vc.data_ptr()),
                               ctypes.c_void_p(ks.data_ptr()), ctypes.c_void_p(vs.data_ptr()),
                               2, 16, None)
    assert st == 2                                                          # head_dim 96
    st = L.kvq_quantize_append(ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                               Hkv * D, Hkv * D, 3, Hkv, D, 0, ctypes.c_void_p(slots.data_ptr()),
                               ctypes.c_void_p(kc.data_ptr()), ctypes.c_void_p(vc.data_ptr()),
                               ctypes.c_void_p(ks.data_ptr()), ctypes.c_void_p(vs.data_ptr()),
                               2, 32, None)
    assert st == 2                                                          # block_size 32
    with pytest.raises(ValueError):                                        # shape mismatch
        kvq.kvq_quantize_append(k, k, slots, kc[:, :, :, :32].contiguous(), vc, ks, vs)


@pytest.mark.parametrize("D,dtype", [(128, "bf16"), (64, "fp16"), (128, "fp16"), (64, "bf16")])
def test_quantize_row_layouts(D, dtype):
    """The append reads 32-byte lane slices when the K and V rows are 16-byte
    aligned (pointers and token strides) and 8-byte slices otherwise: a
    contiguous batch, one with a token stride of Hkv*D + 4 elements and one
    starting 8 bytes into its buffer all write the oracle's codes and scales."""
    T, Hkv = 97, 3
    rng = np.random.default_rng(D + len(dtype))
    x = rng.standard_normal((2, T, Hkv, D)).astype(np.float32) * rng.choice([1e-3, 1, 50], (2, T, Hkv, 1))
    x[:, 5] = 0.0                                  # an all-zero token
    # a token of exact ties: absmax 63.5 gives scale 0.5, and (k + 1/2) * 0.5
    # lies halfway between two codes
    x[:, 7] = ((np.arange(D) % 100) - 50 + 0.5) * 0.5
    x[:, 7, :, 0] = 63.5
    bits = (x.astype(np.float16).view(np.uint16) if dtype == "fp16" else
            torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    qk, sk = oracle.quantize_rows(bits[0], dtype)
    qv, sv = oracle.quantize_rows(bits[1], dtype)
    nb = (T + 15) // 16 + 2
    slots = torch.from_numpy(rng.permutation(nb * 16)[:T].astype(np.int64)).cuda()
    dev = [to_dev(bits[i], dtype) for i in range(2)]
    tdt = dev[0].dtype
    layouts = {"contiguous": dev}
    for name, pad, off in (("token stride + 4", 4, 0), ("8-byte offset", 0, 4)):
        views = []
        for i in range(2):
            buf = torch.zeros(off + T * (Hkv * D + pad), dtype=tdt, device="cuda")
            view = buf[off:].view(T, Hkv * D + pad)[:, :Hkv * D].view(T, Hkv, D)
            view.copy_(dev[i])
            views.append(view)
        layouts[name] = views
    for name, (k, v) in layouts.items():
        kc, vc, ks, vs = kvq.alloc_int8_cache(nb, Hkv, D, "cuda")
        kvq.kvq_quantize_append(k, v, slots, kc, vc, ks, vs)
        blk, o = slots // 16, slots % 16
        assert np.array_equal(kc[blk, :, o].cpu().numpy(), qk), name
        assert np.array_equal(vc[blk, :, o].cpu().numpy(), qv), name
        assert np.array_equal(ks[blk, :, o].cpu().numpy().view(np.uint16), sk), name
        assert np.array_equal(vs[blk, :, o].cpu().numpy().view(np.uint16), sv), name
    assert kvq.kvq_get_error() == (0, 0)
