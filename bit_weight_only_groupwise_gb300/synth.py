"""Seeded synthetic inputs for the groupwise int4/int5 dequant-GEMM.

This module only draws inputs: integer codes, fp16 group scales and bf16
activations, and encodes the codes in the canonical packed byte format that
the library's pack step consumes.  It holds none of the method's arithmetic
(no dequantisation, no products, no sums), so both the CUDA path and the CPU
oracle can be fed from it.

Random numbers come from a counter-based splitmix64 stream: element ``i`` of
tensor ``tid`` under ``seed`` is ``mix64(base(seed, tid) + (i + 1) * GOLDEN)``,
so any element can be recomputed on its own and a [T, K] activation drawn for
T columns is a prefix of the one drawn for more columns.

Distributions (the workloads of the groupwise-int weight format in
"ninfer-3080 docs/performance.md", sections on the small-T kernels and the
A8 prefill routes, and the shapes those sections quote):

* codes: uniform over the 2^b two's-complement values of a b-bit code,
  int4 in [-8, 7], int5 in [-16, 15] (top bits of one draw, unbiased);
* scales: fp16 (round to nearest even) of ``0.002 + 0.01 * |N(0,1)|``, one
  per row per 64 K-columns;
* activations: bf16 (round to nearest even, once, from fp64) of N(0,1); with
  outliers, ``round(0.01 * K)`` input channels chosen once per seed are
  multiplied by 20 for every token before that single rounding -- the pages
  note that activation outliers concentrate in a few input channels.
* normals: Box-Muller on two 53-bit uniforms, cosine branch only.

Canonical packing (the library's input format, see include/qgemm.h):

* int4: row-major, ``ceil(K/2)`` bytes per row; byte j holds code 2j in bits
  0-3 and code 2j+1 in bits 4-7, each as a 4-bit two's-complement field.
* int5: row-major, ``ceil(5K/8)`` bytes per row; an LSB-first bitstream in
  which code k occupies bits 5k .. 5k+4 as a 5-bit two's-complement field.
"""
from __future__ import annotations

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_TID_MUL = 0xD1B54A32D192ED03
_MASK64 = (1 << 64) - 1

# tensor ids; each parent of a multi-parent call adds 16 * parent index
TID_CODES = 1
TID_SCALES = 2
TID_X = 3
TID_OUTLIERS = 4

GROUP = 64


def _mix64_int(z: int) -> int:
    z &= _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def mix64(z: np.ndarray) -> np.ndarray:
    """splitmix64 output function on a uint64 array (wrapping arithmetic)."""
    z = z.astype(np.uint64, copy=True)
    with np.errstate(over="ignore"):
        z ^= z >> np.uint64(30)
        z *= _M1
        z ^= z >> np.uint64(27)
        z *= _M2
        z ^= z >> np.uint64(31)
    return z


def stream_base(seed: int, tid: int) -> int:
    return _mix64_int((seed * 0x9E3779B97F4A7C15) ^ (tid * _TID_MUL))


def draws(seed: int, tid: int, start: int, count: int) -> np.ndarray:
    """uint64 draws ``start .. start+count-1`` of stream (seed, tid)."""
    base = np.uint64(stream_base(seed, tid))
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return mix64(base + idx * GOLDEN)


def uniforms53(z: np.ndarray) -> np.ndarray:
    """53-bit uniforms in [0, 1)."""
    return (z >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normals(seed: int, tid: int, count: int, start: int = 0) -> np.ndarray:
    """N(0,1) draws; normal i uses draws 2i and 2i+1 of the stream."""
    z = draws(seed, tid, 2 * start, 2 * count)
    u1 = 1.0 - uniforms53(z[0::2])          # (0, 1]
    u2 = uniforms53(z[1::2])
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


# ---------------------------------------------------------------- rounding

def fp64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp64 to bf16 once, to nearest even; returns uint16 bit patterns.

    Only for finite values inside bf16's normal range (the generators never
    leave it).  The fp64 significand is rounded to 8 bits, after which the
    value converts to fp32 exactly and its top half is the bf16 pattern.
    """
    x = np.ascontiguousarray(x, dtype=np.float64)
    b = x.view(np.uint64)
    shift = np.uint64(45)                    # 52 - 7 stored bf16 mantissa bits
    lsb = (b >> shift) & np.uint64(1)
    with np.errstate(over="ignore"):
        r = (b + (np.uint64((1 << 44) - 1) + lsb)) & ~np.uint64((1 << 45) - 1)
    f32 = r.view(np.float64).astype(np.float32)   # exact: <= 8 significant bits
    return (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def fp64_to_fp16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp64 to fp16 once, to nearest even (numpy converts directly)."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


# ---------------------------------------------------------------- draws

NVFP4 = 16   # codec id of NVFP4 weights (E2M1 codes, UE4M3 block scales, fp32 tensor scale)
NVFP4_BLOCK = 16
NVFP4_TENSOR_SCALE = 2.0 ** -8 * 1.25   # exact in fp32


def nvfp4_codes(seed: int, tid: int, N: int, K: int) -> np.ndarray:
    """uint8 E2M1 codes [N, K] (0..15), uniform over all sixteen patterns."""
    z = draws(seed, tid, 0, N * K)
    return (z >> np.uint64(60)).astype(np.uint8).reshape(N, K)


def nvfp4_block_scales(seed: int, tid: int, N: int, K: int) -> np.ndarray:
    """uint8 unsigned-E4M3 codes [N, ceil(K/16)]: exponent field uniform in 4..11,
    mantissa uniform (values 2^-3 .. 30)."""
    nb = (K + NVFP4_BLOCK - 1) // NVFP4_BLOCK
    z = draws(seed, tid, 0, N * nb)
    e = 4 + (z >> np.uint64(61)).astype(np.uint8)                  # 4 .. 11
    m = ((z >> np.uint64(58)) & np.uint64(7)).astype(np.uint8)
    return ((e << 3) | m).astype(np.uint8).reshape(N, nb)


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """Raw 4-bit codes [N, K] two per byte: column 2j in bits 0-3, 2j+1 in bits 4-7."""
    codes = np.asarray(codes, np.uint8)
    N, K = codes.shape
    if K % 2:
        codes = np.concatenate([codes, np.zeros((N, 1), np.uint8)], axis=1)
    return ((codes[:, 0::2] & 0x0F) | ((codes[:, 1::2] & 0x0F) << 4)).astype(np.uint8)


def uniform_codes(seed: int, tid: int, N: int, K: int, bits: int) -> np.ndarray:
    """int8 codes [N, K], uniform over the b-bit two's-complement range; for
    bits = 8, uint8 E4M3 codes uniform over the 254 that are not NaN (a NaN
    code S.1111.111 is replaced by S.1111.110, the largest finite value)."""
    if bits == 8:
        z = draws(seed, tid, 0, N * K)
        u = (z >> np.uint64(56)).astype(np.uint8)
        u[(u & 0x7F) == 0x7F] ^= np.uint8(1)
        return u.reshape(N, K)
    if bits not in (4, 5):
        raise ValueError("bits must be 4, 5 or 8")
    z = draws(seed, tid, 0, N * K)
    u = (z >> np.uint64(64 - bits)).astype(np.int16)
    return (u - (1 << (bits - 1))).astype(np.int8).reshape(N, K)


def group_scales(seed: int, tid: int, N: int, K: int) -> np.ndarray:
    """fp16 bit patterns [N, ceil(K/64)] of 0.002 + 0.01*|N(0,1)|."""
    G = (K + GROUP - 1) // GROUP
    n = normals(seed, tid, N * G)
    return fp64_to_fp16_bits(0.002 + 0.01 * np.abs(n)).reshape(N, G)


def outlier_channels(seed: int, K: int, tid: int = TID_OUTLIERS) -> np.ndarray:
    """The round(0.01*K) channels chosen for a seed, sorted ascending."""
    m = int(np.floor(0.01 * K + 0.5))
    keys = draws(seed, tid, 0, K)
    order = np.argsort(keys, kind="stable")
    return np.sort(order[:m])


def activations(seed: int, T: int, K: int, outliers: bool, tid: int = TID_X) -> np.ndarray:
    """bf16 bit patterns [T, K]: N(0,1), outlier channels x20, one rounding."""
    x = normals(seed, tid, T * K).reshape(T, K)
    if outliers:
        x[:, outlier_channels(seed, K)] *= 20.0
    return fp64_to_bf16_bits(x).reshape(T, K)


# ---------------------------------------------------------------- canonical packing

def row_bytes(K: int, bits: int) -> int:
    return (K * bits + 7) // 8


def pack_canonical(codes: np.ndarray, bits: int) -> np.ndarray:
    """Encode codes [N, K] in the canonical packed format (uint8 [N, row_bytes]);
    fp8 codes are their own canonical bytes."""
    codes = np.asarray(codes)
    N, K = codes.shape
    if bits == 8:
        return np.ascontiguousarray(codes, dtype=np.uint8).copy()
    lo = -(1 << (bits - 1))
    hi = (1 << (bits - 1)) - 1
    if codes.size and (codes.min() < lo or codes.max() > hi):
        raise ValueError(f"codes outside the {bits}-bit range")
    field = (codes.astype(np.int16) & ((1 << bits) - 1)).astype(np.uint8)
    if bits == 4:
        if K % 2:
            field = np.concatenate([field, np.zeros((N, 1), np.uint8)], axis=1)
        return (field[:, 0::2] | (field[:, 1::2] << 4)).astype(np.uint8)
    # int5: LSB-first bitstream per row
    bitarr = np.zeros((N, row_bytes(K, 5) * 8), np.uint8)
    for b in range(5):
        bitarr[:, np.arange(K) * 5 + b] = (field >> b) & 1
    return np.packbits(bitarr, axis=1, bitorder="little")


# ---------------------------------------------------------------- workloads

def weights(seed: int, N: int, K: int, bits: int, parent: int = 0) -> dict:
    """Codes, their canonical packing and group scales of one weight matrix
    (NVFP4, bits = 16: E2M1 codes, UE4M3 block scales and the tensor scale)."""
    off = 16 * parent
    if bits == NVFP4:
        codes = nvfp4_codes(seed, TID_CODES + off, N, K)
        return {"bits": bits, "N": N, "K": K, "codes": codes, "packed": pack_nibbles(codes),
                "scales": nvfp4_block_scales(seed, TID_SCALES + off, N, K), "tscale": NVFP4_TENSOR_SCALE}
    codes = uniform_codes(seed, TID_CODES + off, N, K, bits)
    return {
        "bits": bits,
        "N": N,
        "K": K,
        "codes": codes,
        "packed": pack_canonical(codes, bits),
        "scales": group_scales(seed, TID_SCALES + off, N, K),
    }


# Projection shapes of a 5120-hidden, 27B-class model quoted on the
# "ninfer-3080 docs/performance.md" page (small-T kernel table and the
# A8 prefill route table); T values are the decode, verify, batched-decode and
# prefill widths those sections discuss.
CONFIGS = {
    "tiny": dict(parents=[(256, 4)], K=512, Ts=[1], outliers=False),
    "decode": dict(parents=[(5120, 4)], K=6144, Ts=[1, 2, 4, 8], outliers=True),
    "batched": dict(parents=[(12288, 4)], K=5120, Ts=[16, 32, 64, 256], outliers=True),
    "multi": dict(parents=[(4096, 4), (12288, 5)], K=5120, Ts=[4, 16, 64], outliers=True),
    "prefill_a": dict(parents=[(7168, 4)], K=5120, Ts=[256, 1024, 4096], outliers=True),
    "prefill_b": dict(parents=[(5120, 4)], K=6144, Ts=[256, 1024, 4096], outliers=True),
    # fused outputs at decode widths: the Q5 [5120, 6144] LinearAdd of the
    # attention o_proj / GDN out_proj, and the Q4 gate_up projection (34816 x
    # 5120) as a SwiGLU pair of two 17408-row matrices (parents 0 and 1)
    "linear_add": dict(parents=[(5120, 5)], K=6144, Ts=[1, 2, 4, 8], outliers=True, epilogue="add"),
    "swiglu": dict(parents=[(17408, 4), (17408, 4)], K=5120, Ts=[1, 2, 4, 8], outliers=True, epilogue="swiglu"),
    # the decode shape with FP8 (E4M3) weights at decode and verify widths
    "decode_fp8": dict(parents=[(5120, 8)], K=6144, Ts=[1, 2, 4, 8], outliers=True),
    "prefill_fp8": dict(parents=[(7168, 8)], K=5120, Ts=[256, 1024, 4096], outliers=True),
    # NVFP4 weights at decode and prefill widths
    "decode_nvfp4": dict(parents=[(5120, NVFP4)], K=6144, Ts=[1, 2, 4, 8], outliers=True),
    "prefill_nvfp4": dict(parents=[(7168, NVFP4)], K=5120, Ts=[256, 1024, 4096], outliers=True),
    # K / 64 = 90 groups, not a multiple of 8: the small-T route's ring kernel
    "decode_ring": dict(parents=[(5120, 4)], K=5760, Ts=[1, 8, 16], outliers=True),
}


def workload(name: str, T: int, seed: int = 0) -> dict:
    """All inputs of one named workload at width T: ``parents`` and ``x``."""
    cfg = CONFIGS[name]
    K = cfg["K"]
    parents = [weights(seed, N, K, bits, parent=i) for i, (N, bits) in enumerate(cfg["parents"])]
    x = activations(seed, T, K, cfg["outliers"])
    return {"name": name, "K": K, "T": T, "parents": parents, "x": x}
