"""CPU oracle of the Lynx split-stream KV codec and of decode attention.

TEST INFRASTRUCTURE ONLY.  The product library (``split_stream_kv_gb300``)
never imports this package; only ``tests/``, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline leg do.  The arithmetic lives in the plain C file
``lynx_oracle.c`` (compiled with ``-ffp-contract=off -fno-fast-math``); this
module builds it, loads it with ctypes and wraps it for numpy arrays.  A few
closed-form size formulas from the pages are written here in Python.

Sources, cited by page title and section:
  [Review] "Lynx: Progressive Speculative KV Cache Transfer for Disaggregated
           LLM Inference" (technical review of the paper).
  [Digest] "Lynx: Progressive Speculative Quantization for accelerating KV
           Transfer in Long-Context Inference" (paper digest).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lynx_oracle.c")
_LIB = os.path.join(_HERE, "liblynx_oracle.so")
_lock = threading.Lock()
_lib = None

EPS = 1e-6  # the pages leave eps open; float32 1e-6 on both sides


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _bind(lib):
    """Declare the C signatures on a loaded oracle library."""
    P, I64, I, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    lib.oracle_compand_y.argtypes = [F, F]
    lib.oracle_compand_y.restype = ctypes.c_double
    lib.oracle_round_code.argtypes = [F, F]
    lib.oracle_round_code.restype = I
    lib.oracle_expand.argtypes = [I, F]
    lib.oracle_expand.restype = F
    lib.oracle_stage4_literal.argtypes = [I, I, P]
    lib.oracle_stage4_literal.restype = None
    lib.oracle_code8.argtypes = [I, I]
    lib.oracle_code8.restype = I
    lib.oracle_anchor_nibble.argtypes = [I]
    lib.oracle_anchor_nibble.restype = I
    lib.oracle_residual_nibble.argtypes = [I]
    lib.oracle_residual_nibble.restype = I
    lib.oracle_f32_to_bf16.argtypes = [F]
    lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
    lib.oracle_f32_to_bf16_array.argtypes = [P, P, I64]
    lib.oracle_f32_to_bf16_array.restype = None
    lib.oracle_encode_block.argtypes = [P, I64, I, I, I, F, P, P, P]
    lib.oracle_encode_block.restype = I
    lib.oracle_encode_range.argtypes = [P, I64, I64, I, I, I, I, F, P, P, P,
                                        I64, I64]
    lib.oracle_encode_range.restype = I
    lib.oracle_decode_block.argtypes = [P, P, P, I, I, I, F, P, I64]
    lib.oracle_decode_block.restype = I
    lib.oracle_decode_range.argtypes = [P, P, P, I64, I64, I, I, I, I, F, P,
                                        I64, I64]
    lib.oracle_decode_range.restype = I
    lib.oracle_attention_row.argtypes = [P, P, P, I64, I, I64, P]
    lib.oracle_attention_row.restype = None
    lib.oracle_attention_row_tail.argtypes = [P, P, P, I64, P, P, I, I, I64, I64, P]
    lib.oracle_attention_row_tail.restype = None
    lib.oracle_spec_verify.argtypes = [P, P, P, P, ctypes.c_uint32, I, I64, P]
    lib.oracle_spec_verify.restype = I
    lib.oracle_spec_verify_batch.argtypes = [P, P, P, P, P, I, I, I64, P, P]
    lib.oracle_spec_verify_batch.restype = None
    lib.oracle_split_bits.argtypes = [P, P, I64, I, I, P, P]
    lib.oracle_split_bits.restype = I
    lib.oracle_decode_anchor_bits_range.argtypes = [P, P, I64, I64, I, I, I, I, F, I, P]
    lib.oracle_decode_anchor_bits_range.restype = I
    lib.oracle_a1_encode_range.argtypes = [P, I64, I64, I, I, I, F, P, P, P]
    lib.oracle_a1_encode_range.restype = I
    lib.oracle_a1_decode_range.argtypes = [P, P, P, I64, I64, I, I, I, F, P]
    lib.oracle_a1_decode_range.restype = I
    lib.oracle_int_encode_rows.argtypes = [P, I64, I, I, P, P]
    lib.oracle_int_encode_rows.restype = I
    lib.oracle_int_decode_rows.argtypes = [P, P, I64, I, I, P]
    lib.oracle_int_decode_rows.restype = I
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        _lib = _bind(ctypes.CDLL(_LIB))
        return _lib


class using_library:
    """Context manager: route every oracle call through another compiled
    copy of lynx_oracle.c (the tests build deliberately broken copies to show
    that the pins catch them)."""

    def __init__(self, path: str):
        self.lib = _bind(ctypes.CDLL(path))

    def __enter__(self):
        global _lib
        _load()
        self.saved = _lib
        _lib = self.lib
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def compile_variant(src_text: str, out_path: str) -> str:
    """Compile C source text with the oracle's flags into out_path."""
    c_path = out_path[:-3] + ".c"
    with open(c_path, "w") as f:
        f.write(src_text)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-o", out_path, c_path, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True)
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


# ------------------------------------------------------------ scalar pieces

def compand_y(a: float, alpha: float) -> float:
    """Eq. 7 value Y in float64 from float32 |X_final| [Review, Stage 3]."""
    return _load().oracle_compand_y(a, alpha)


def round_code(a: float, alpha: float) -> int:
    """I = Round(Y) in 0..127 [Review, Stage 3]."""
    return _load().oracle_round_code(a, alpha)


def expand(I: int, alpha: float) -> float:
    """float32(((1+alpha)^(I/127) - 1)/alpha) [Review, Eq. 14/15]."""
    return _load().oracle_expand(I, alpha)


def expand_table(alpha: float) -> np.ndarray:
    return np.array([expand(i, alpha) for i in range(128)], dtype=np.float32)


def stage4_literal(I: int, S: int) -> dict:
    """Stage 4 exactly as printed: I_bias, V_mag, V_recon, V_res, Q_anc
    [Review, Stage 4, Eq. 9]."""
    out = (ctypes.c_int * 5)()
    _load().oracle_stage4_literal(I, S, ctypes.cast(out, ctypes.c_void_p))
    return dict(I_bias=out[0], V_mag=out[1], V_recon=out[2], V_res=out[3],
                Q_anc=out[4])


def code8(I: int, S: int) -> int:
    """Eq. 9 on the full magnitude, as an 8-bit two's-complement pattern."""
    return _load().oracle_code8(I, S)


def anchor_nibble(c8: int) -> int:
    return _load().oracle_anchor_nibble(c8)


def residual_nibble(c8: int) -> int:
    return _load().oracle_residual_nibble(c8)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even, NaN kept
    a NaN: the oracle's oracle_f32_to_bf16 applied elementwise."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    _load().oracle_f32_to_bf16_array(_ptr(x), _ptr(out), x.size)
    return out


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32)
            << 16).view(np.float32)


# ------------------------------------------------------------ codec

def meta_rows(P: int, C: int) -> int:
    """2 + 2P/C float32 rows of D per page block [Review, Stage 1 and 2]."""
    return 2 + 2 * (P // C)


def encode_block(x_bits: np.ndarray, C: int, alpha: float):
    """Algorithm 1 on one block x_bits[P][D] (uint16 BF16 bits)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    P, D = x.shape
    anc = np.zeros((P, D // 2), np.uint8)
    res = np.zeros((P, D // 2), np.uint8)
    meta = np.zeros((meta_rows(P, C), D), np.float32)
    rc = _load().oracle_encode_block(_ptr(x), D, P, D, C, alpha, _ptr(anc),
                                     _ptr(res), _ptr(meta))
    if rc:
        raise ValueError("oracle_encode_block: bad arguments")
    return anc, res, meta


def _split(n: int, parts: int):
    parts = max(1, min(parts, n))
    step = (n + parts - 1) // parts
    return [(i, min(n, i + step)) for i in range(0, n, step)]


def encode(kv_bits: np.ndarray, P: int, C: int, alpha: float,
           threads: int = 1, block_range=None):
    """Encode kv_bits[B][L][H][D] (uint16 BF16 bits).  Returns
    (anchor[B][NB][H][P][D/2], residual, meta[B][NB][H][2+2P/C][D])."""
    kv = np.ascontiguousarray(kv_bits, dtype=np.uint16)
    B, L, H, D = kv.shape
    NB = L // P
    anc = np.zeros((B, NB, H, P, D // 2), np.uint8)
    res = np.zeros_like(anc)
    meta = np.zeros((B, NB, H, meta_rows(P, C), D), np.float32)
    lo, hi = block_range if block_range is not None else (0, B * NB * H)
    lib = _load()

    def run(rng):
        rc = lib.oracle_encode_range(_ptr(kv), B, L, H, D, P, C, alpha,
                                     _ptr(anc), _ptr(res), _ptr(meta),
                                     rng[0], rng[1])
        if rc:
            raise ValueError("oracle_encode_range: bad arguments")

    chunks = [(a + lo, b + lo) for a, b in _split(hi - lo, threads)]
    if threads <= 1 or len(chunks) == 1:
        for c in chunks:
            run(c)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(run, chunks))
    return anc, res, meta


def decode_block(anc: np.ndarray, res, meta: np.ndarray, C: int,
                 alpha: float) -> np.ndarray:
    """Decode one block; res=None gives the Anchor-only reconstruction."""
    anc = np.ascontiguousarray(anc, dtype=np.uint8)
    P = anc.shape[0]
    D = anc.shape[1] * 2
    meta = np.ascontiguousarray(meta, dtype=np.float32)
    out = np.zeros((P, D), np.float32)
    rp = None
    if res is not None:
        res = np.ascontiguousarray(res, dtype=np.uint8)
        rp = _ptr(res)
    rc = _load().oracle_decode_block(_ptr(anc), rp, _ptr(meta), P, D, C, alpha,
                                     _ptr(out), D)
    if rc:
        raise ValueError("oracle_decode_block: bad arguments")
    return out


def decode(anc: np.ndarray, res, meta: np.ndarray, L: int, P: int, C: int,
           alpha: float, threads: int = 1, block_range=None) -> np.ndarray:
    """Decode streams laid out as encode() returns them to float32
    [B][L][H][D]; res=None gives the Anchor-only reconstruction."""
    anc = np.ascontiguousarray(anc, dtype=np.uint8)
    B, NB, H, _, half = anc.shape
    D = half * 2
    meta = np.ascontiguousarray(meta, dtype=np.float32)
    out = np.zeros((B, L, H, D), np.float32)
    rp = None
    if res is not None:
        res = np.ascontiguousarray(res, dtype=np.uint8)
        rp = _ptr(res)
    lib = _load()
    lo, hi = block_range if block_range is not None else (0, B * NB * H)

    def run(rng):
        rc = lib.oracle_decode_range(_ptr(anc), rp, _ptr(meta), B, L, H, D, P,
                                     C, alpha, _ptr(out), rng[0], rng[1])
        if rc:
            raise ValueError("oracle_decode_range: bad arguments")

    chunks = [(a + lo, b + lo) for a, b in _split(hi - lo, threads)]
    if threads <= 1 or len(chunks) == 1:
        for c in chunks:
            run(c)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(run, chunks))
    return out


# ------------------------------------------------------------ attention

def attention_row(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """float64 softmax(q K^T / sqrt(D)) V for one query row [Review, Eq. 1].
    q[D], K[L][D], V[L][D] as float32 (the values the attention sees)."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    K = np.ascontiguousarray(K, dtype=np.float32)
    V = np.ascontiguousarray(V, dtype=np.float32)
    L, D = K.shape
    out = np.zeros(D, np.float64)
    _load().oracle_attention_row(_ptr(q), _ptr(K), _ptr(V), L, D, D, _ptr(out))
    return out


def attention_row_tail(q: np.ndarray, K: np.ndarray, V: np.ndarray, Kt: np.ndarray,
                       Vt: np.ndarray, n_tail: int) -> np.ndarray:
    """float64 attention of the verification row of draft position n_tail - 1
    over the L cached tokens K, V and the draft's own tokens Kt[:n_tail],
    Vt[:n_tail] [Review, Mechanism 3, single parallel verification pass;
    Eq. 1].  All inputs float32 (the values the attention sees)."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    K = np.ascontiguousarray(K, dtype=np.float32)
    V = np.ascontiguousarray(V, dtype=np.float32)
    Kt = np.ascontiguousarray(Kt, dtype=np.float32)
    Vt = np.ascontiguousarray(Vt, dtype=np.float32)
    L, D = K.shape
    if not 0 <= n_tail <= Kt.shape[0]:
        raise ValueError("n_tail out of range")
    out = np.zeros(D, np.float64)
    _load().oracle_attention_row_tail(_ptr(q), _ptr(K), _ptr(V), L, _ptr(Kt), _ptr(Vt),
                                      n_tail, D, D, D, _ptr(out))
    return out


def spec_verify(p: np.ndarray, q: np.ndarray, s: np.ndarray, u: np.ndarray,
                r: np.ndarray):
    """Speculative verification and correction [Review, Mechanism 3, Eq. 10,
    Eq. 11] for a batch: p [batch][T+1][V], q [batch][T][V] float32
    distributions, s [batch][T] draft tokens, u [batch][T] uniforms, r [batch]
    uint32.  Returns (n_accepted [batch], next_token [batch]) as int32."""
    p = np.ascontiguousarray(p, dtype=np.float32)
    q = np.ascontiguousarray(q, dtype=np.float32)
    s = np.ascontiguousarray(s, dtype=np.int32)
    u = np.ascontiguousarray(u, dtype=np.float32)
    r = np.ascontiguousarray(r, dtype=np.uint32)
    batch, T1, V = p.shape
    T = T1 - 1
    if q.shape != (batch, T, V) or s.shape != (batch, T) or u.shape != (batch, T):
        raise ValueError("spec_verify: shapes")
    k = np.empty(batch, np.int32)
    tok = np.empty(batch, np.int32)
    _load().oracle_spec_verify_batch(_ptr(p), _ptr(q), _ptr(s), _ptr(u), _ptr(r), batch, T, V,
                                     _ptr(k), _ptr(tok))
    return k, tok


# ------------------------------------------------------------ variants

def split_bits(anc4: np.ndarray, res4: np.ndarray, k: int):
    """Re-split 4+4 streams [..][P][D/2] into a k + (8-k) split: returns the
    Anchor [..][P][D*k/8] and Residual [..][P][D*(8-k)/8] streams."""
    lib = _load()
    a = np.ascontiguousarray(anc4, dtype=np.uint8)
    r = np.ascontiguousarray(res4, dtype=np.uint8)
    D = a.shape[-1] * 2
    rows = a.size // (D // 2)
    ak = np.zeros(a.shape[:-1] + (D * k // 8,), dtype=np.uint8)
    rk = np.zeros(a.shape[:-1] + (D * (8 - k) // 8,), dtype=np.uint8)
    rc = lib.oracle_split_bits(_ptr(a), _ptr(r), rows, D, k, _ptr(ak), _ptr(rk))
    if rc:
        raise ValueError("oracle_split_bits: bad arguments")
    return ak, rk


def decode_anchor_bits(ak: np.ndarray, meta: np.ndarray, L: int, P: int, C: int, alpha: float,
                       k: int) -> np.ndarray:
    """Anchor-only decode of a k-bit Anchor stream [B][NB][H][P][D*k/8]."""
    lib = _load()
    a = np.ascontiguousarray(ak, dtype=np.uint8)
    m = np.ascontiguousarray(meta, dtype=np.float32)
    B, NB, H = a.shape[:3]
    D = a.shape[-1] * 8 // k
    out = np.zeros((B, L, H, D), dtype=np.float32)
    rc = lib.oracle_decode_anchor_bits_range(_ptr(a), _ptr(m), B, L, H, D, P, C, alpha, k,
                                             _ptr(out))
    if rc:
        raise ValueError("oracle_decode_anchor_bits_range: bad arguments")
    return out


def a1_encode(kv_bits: np.ndarray, P: int, alpha: float = 100.0):
    """The Appendix A.1 variant of a bf16 tensor [B][L][H][D] (uint16 bit
    patterns): anchor, residual [B][NB][H][P][D/2] and meta
    [B][NB][H][1 + P/16][D]."""
    lib = _load()
    x = np.ascontiguousarray(kv_bits, dtype=np.uint16)
    B, L, H, D = x.shape
    NB = L // P
    anc = np.zeros((B, NB, H, P, D // 2), np.uint8)
    res = np.zeros_like(anc)
    meta = np.zeros((B, NB, H, 1 + P // 16, D), np.float32)
    rc = lib.oracle_a1_encode_range(_ptr(x), B, L, H, D, P, alpha, _ptr(anc), _ptr(res),
                                    _ptr(meta))
    if rc:
        raise ValueError("oracle_a1_encode_range: bad arguments")
    return anc, res, meta


def a1_decode(anc: np.ndarray, res, meta: np.ndarray, L: int, P: int,
              alpha: float = 100.0) -> np.ndarray:
    """Decode of the A.1 variant (res None: Anchor only) to float32
    [B][L][H][D]."""
    lib = _load()
    a = np.ascontiguousarray(anc, dtype=np.uint8)
    r = None if res is None else np.ascontiguousarray(res, dtype=np.uint8)
    m = np.ascontiguousarray(meta, dtype=np.float32)
    B, NB, H = a.shape[:3]
    D = a.shape[-1] * 2
    out = np.zeros((B, L, H, D), np.float32)
    rc = lib.oracle_a1_decode_range(_ptr(a), None if r is None else _ptr(r), _ptr(m), B, L, H, D,
                                    P, alpha, _ptr(out))
    if rc:
        raise ValueError("oracle_a1_decode_range: bad arguments")
    return out


def int_encode(kv_bits: np.ndarray, bits: int):
    """Linear INT-`bits` baseline (Eq. 4) of a bf16 tensor [..][D] (uint16
    bit patterns): codes [..][D*bits/8] uint8 and meta [..][2] float32."""
    lib = _load()
    x = np.ascontiguousarray(kv_bits, dtype=np.uint16)
    D = x.shape[-1]
    rows = x.size // D
    codes = np.zeros(x.shape[:-1] + (D * bits // 8,), dtype=np.uint8)
    meta = np.zeros(x.shape[:-1] + (2,), dtype=np.float32)
    rc = lib.oracle_int_encode_rows(_ptr(x), rows, D, bits, _ptr(codes), _ptr(meta))
    if rc:
        raise ValueError("oracle_int_encode_rows: bad arguments")
    return codes, meta


def int_decode(codes: np.ndarray, meta: np.ndarray, bits: int) -> np.ndarray:
    lib = _load()
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    m = np.ascontiguousarray(meta, dtype=np.float32)
    D = c.shape[-1] * 8 // bits
    rows = c.size // (D * bits // 8)
    out = np.zeros(c.shape[:-1] + (D,), dtype=np.float32)
    rc = lib.oracle_int_decode_rows(_ptr(c), _ptr(m), rows, D, bits, _ptr(out))
    if rc:
        raise ValueError("oracle_int_decode_rows: bad arguments")
    return out


def vnmse(approx: np.ndarray, ref: np.ndarray) -> float:
    """Normalised mean-square error of attention outputs (the metric of the
    pages' accuracy table, [Review], Mechanism 3 "Why is the acceptance rate
    high?"): sum |o - o_ref|^2 / sum |o_ref|^2 over all outputs, float64."""
    a = np.asarray(approx, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    return float(np.sum((a - r) ** 2) / np.sum(r ** 2))


def attention_rows(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """attention_row for every (sequence, query token, query head): q
    [batch][T][H_q][D], K, V [batch][L][H_kv][D] float32 (GQA: query head h
    reads KV head h // (H_q/H_kv)); float64 out [batch][T][H_q][D]."""
    batch, T, Hq, D = q.shape
    Hkv = K.shape[2]
    G = Hq // Hkv
    out = np.zeros((batch, T, Hq, D), dtype=np.float64)
    for b in range(batch):
        for h in range(Hkv):
            Kh = np.ascontiguousarray(K[b, :, h, :], dtype=np.float32)
            Vh = np.ascontiguousarray(V[b, :, h, :], dtype=np.float32)
            for t in range(T):
                for g in range(G):
                    out[b, t, h * G + g] = attention_row(q[b, t, h * G + g], Kh, Vh)
    return out


# ------------------------------------------------------------ size formulas

def kv_size_bytes(k_factor: int, L: int, D: int, n_layers: int,
                  precision_bytes: int) -> int:
    """Size_KV = K_factor * L * D * N_layers * Precision, D = H_heads*D_head
    [Review, Prerequisites, Eq. 2]."""
    return k_factor * L * D * n_layers * precision_bytes


def metadata_scalars(H: int, P: int, C: int) -> int:
    """H * (2 + 2P/C) scalars per page block [Review, "Why Not Global Grouped
    Quantization?"]."""
    return H * (2 + 2 * (P // C))


def effective_bins(B: int, ratio_local_to_global: float) -> float:
    """Bins_eff ~ 2^B * m_i / m [Review, Prerequisites, Eq. 5]."""
    return (2 ** B) * ratio_local_to_global


def anchor_ratio(alpha: float) -> float:
    """Ratio of consecutive Anchor buckets (1+alpha)^(16/127): the geometric
    interval of the Anchor ("effective exponentiation (1+alpha)^q_anc",
    [Digest, Method])."""
    return (1.0 + alpha) ** (16.0 / 127.0)


# ------------------------------------------------------------ request format

def stream_bytes(B: int, L: int, H: int, P: int, C: int, D: int = 128):
    """Bytes of the Anchor, Residual and meta streams: 4 bits per element for
    each code stream [Review, Implementation Notes: two 4-bit values per
    uint8], (2 + 2P/C) float32 rows of D per page block (the metadata above)."""
    elems = B * L * H * D
    return elems // 2, elems // 2, B * (L // P) * metadata_scalars(H, P, C) * D * 4


def request_header(B: int, L: int, H: int, P: int, C: int, alpha: float,
                   with_residual: bool = True, D: int = 128, version: int = 1,
                   sizes=None) -> bytes:
    """The 128-byte header of a serialized request, written out field by
    field: the Anchor stream and its metadata first, so the Anchor phase is
    one contiguous range ("Q_anc and metadata contiguous", [Review],
    Implementation Notes), then the Residual stream.  The last field is the
    CRC-32 (zlib's) of the 124 bytes before it.  `sizes` overrides the
    stream sizes (to build inconsistent headers for tests)."""
    import struct
    import zlib
    a, r, m = sizes if sizes is not None else stream_bytes(B, L, H, P, C, D)
    if not with_residual and sizes is None:
        r = 0
    a_off = 128
    m_off = a_off + a
    r_off = m_off + m
    body = struct.pack("<8sIIqqiiiifIQQQQQQQIII", b"LYNXKV\x00\x01", version, 128, B, L, H, D,
                       P, C, alpha, 1 if with_residual else 0, a_off, a, m_off, m, r_off, r,
                       r_off + r, 0, 0, 0)
    assert len(body) == 124
    return body + struct.pack("<I", zlib.crc32(body) & 0xFFFFFFFF)


__all__ = [
    "EPS", "build", "compand_y", "round_code", "expand", "expand_table",
    "stage4_literal", "code8", "anchor_nibble", "residual_nibble",
    "f32_to_bf16_bits", "bf16_bits_to_f32", "meta_rows", "encode_block",
    "encode", "decode_block", "decode", "attention_row", "kv_size_bytes",
    "metadata_scalars", "effective_bins", "anchor_ratio", "stream_bytes", "request_header",
    "split_bits", "decode_anchor_bits", "int_encode", "int_decode", "vnmse", "attention_rows",
    "a1_encode", "a1_decode",
]
