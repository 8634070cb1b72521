"""ctypes binding of liblynx.so (include/lynx.h), one Python function per C
entry point with the same name.  Only argument marshalling happens here:
tensors become device pointers and sizes, the current CUDA stream is passed
along, and output tensors are allocated with torch when the caller gives none.
There is no CPU path: non-CUDA tensors are rejected.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# LYNX_LIBRARY=checked selects the checked build (liblynx_checked.so: kernels
# that verify their index arithmetic and report a failed check through
# lynx_device_errors); the default is the regular build.
LIB_PATH = os.path.join(_HERE, "liblynx_checked.so" if os.environ.get("LYNX_LIBRARY") == "checked"
                        else "liblynx.so")

LYNX_OK, LYNX_EINVAL, LYNX_ESHAPE, LYNX_EUNSUPPORTED, LYNX_ECUDA, LYNX_EWORKSPACE = (
    0, -1, -2, -3, -4, -5)
LYNX_ANCHOR, LYNX_FULL = 0, 1
LYNX_OUT_BF16, LYNX_OUT_FP32 = 0, 1

_lib = None


class LynxError(RuntimeError):
    def __init__(self, code: int, what: str, detail: str):
        super().__init__(f"{what}: {detail} ({code})")
        self.code = code


def lib() -> ctypes.CDLL:
    """Load liblynx.so (build it first with split_stream_kv_gb300._build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "split_stream_kv_gb300._build.build()")
    L = ctypes.CDLL(LIB_PATH)
    P, I64, I, F, SZ = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                        ctypes.c_size_t)
    PSZ = ctypes.POINTER(ctypes.c_size_t)
    sig = {
        "lynx_encoded_sizes": ([I64, I64, I, I, I, I, PSZ, PSZ, PSZ], I),
        "lynx_encode": ([P, I64, I64, I, I, I, I, F, P, P, P, P], I),
        "lynx_decode_anchor": ([P, P, I64, I64, I, I, I, I, F, P, I, P], I),
        "lynx_decode_full": ([P, P, P, I64, I64, I, I, I, I, F, P, I, P], I),
        "lynx_attn_workspace_bytes": ([I, I, I, I64, I, I, I, PSZ], I),
        "lynx_attn_decode": ([P, I, I, I, P, P, P, P, P, P, I64, I, I, I, I, F, I, P, P, SZ, P],
                             I),
        "lynx_attn_decode_tail": ([P, I, I, I, P, P, P, P, P, P, I64, I, I, I, I, F, I, P, P, P, P,
                                   SZ, P], I),
        "lynx_attn_decode_paged": ([P, I, I, I, P, P, P, P, P, P, P, I64, I64, I, I, I, I, F, I,
                                    P, P, P, P, SZ, P], I),
        "lynx_encode_paged": ([P, I64, I64, I, I, I, I, F, P, I64, P, P, P, P], I),
        "lynx_decode_paged": ([P, P, P, P, I64, I64, I64, I, I, I, I, F, I, P, I, P], I),
        "lynx_device_errors": ([ctypes.POINTER(ctypes.c_uint)], I),
        "lynx_spec_verify": ([P, P, P, P, P, I, I, I64, P, P, P], I),
        "lynx_attn_decode_noalloc": ([P, I, I, I, P, P, P, P, P, P, I64, I, I, I, I, F, I, P, P],
                                     I),
        "lynx_split_plan": ([I64, I64, I, I, I, I, I64, I, I, P, I64,
                             ctypes.POINTER(ctypes.c_int64)], I),
        "lynx_split_receive": ([P, P, P, P, P, P, I64, I64, I, I, I, I, F, I64, P, I, P, P, P,
                                P, P], I),
        "lynx_split_send": ([P, I64, I64, I, I, I, I, F, P, P, P, P, P, P, I64, P, P, P, P], I),
        "lynx_header_init": ([P, I64, I64, I, I, I, I, F, I], I),
        "lynx_header_check": ([P], I),
        "lynx_int_encode": ([P, I64, I, I, P, P, P], I),
        "lynx_int_decode": ([P, P, I64, I, I, P, I, P], I),
        "lynx_split_bits": ([P, P, I64, I, I, P, P, P], I),
        "lynx_join_bits": ([P, P, I64, I, I, P, P, P], I),
        "lynx_decode_anchor_bits": ([P, P, I64, I64, I, I, I, I, F, I, P, I, P], I),
        "lynx_a1_encode": ([P, I64, I64, I, I, I, F, P, P, P, P], I),
        "lynx_a1_decode": ([P, P, P, I64, I64, I, I, I, F, P, I, P], I),
        "lynx_wait_selftest": ([ctypes.c_uint64, I, P, P], I),
        "lynx_compander_thresholds": ([F, P], I),
        "lynx_expand_table": ([F, P], I),
        "lynx_compander_selfcheck": ([F, P, P], I),
        "lynx_wait_timeouts": ([ctypes.POINTER(ctypes.c_uint)], I),
        "lynx_status_string": ([I], ctypes.c_char_p),
        "lynx_last_error": ([], ctypes.c_char_p),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _lib = L
    return L


def _check(rc: int, what: str):
    if rc != LYNX_OK:
        detail = lib().lynx_last_error().decode(errors="replace")
        raise LynxError(rc, what, detail)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("lynx: tensors must be contiguous CUDA tensors")


def _expect(t, shape, dtype, device, what):
    """The C ABI sees pointers only: a caller's tensor of the wrong size or
    type would be read or written out of bounds on the device, so every
    tensor is checked against the sizes the call implies before it is
    passed."""
    if t is None:
        raise ValueError(f"{what} is required")
    if t.dtype != dtype or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{what}: expected {dtype} of shape {tuple(shape)}, got {t.dtype} "
                         f"of shape {tuple(t.shape)}")
    if t.device != device:
        raise ValueError(f"{what}: on {t.device}, expected {device}")


# ----------------------------------------------------------------- codec

def lynx_encoded_sizes(B: int, L: int, H_kv: int, D: int, page: int, C: int):
    a, r, m = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().lynx_encoded_sizes(B, L, H_kv, D, page, C, ctypes.byref(a), ctypes.byref(r),
                                    ctypes.byref(m)), "lynx_encoded_sizes")
    return a.value, r.value, m.value


def stream_shapes(B: int, L: int, H_kv: int, D: int, page: int, C: int):
    """Tensor shapes of (anchor, residual, meta) for a kv[B][L][H_kv][D]."""
    NB = L // page
    codes = (B, NB, H_kv, page, D // 2)
    return codes, codes, (B, NB, H_kv, 2 + 2 * (page // C), D)


def lynx_encode(kv: torch.Tensor, page: int, C: int, alpha: float, anchor=None, residual=None,
                meta=None):
    """Encode kv[B][L][H_kv][D] (bf16, CUDA).  Returns (anchor, residual, meta)."""
    _need_cuda(kv, anchor, residual, meta)
    if kv.dtype != torch.bfloat16 or kv.dim() != 4:
        raise ValueError("lynx_encode: kv must be a 4-D bfloat16 tensor")
    B, L, H, D = kv.shape
    ca, cr, cm = stream_shapes(B, L, H, D, page, C)
    dev = kv.device
    if anchor is None:
        anchor = torch.empty(ca, dtype=torch.uint8, device=dev)
    if residual is None:
        residual = torch.empty(cr, dtype=torch.uint8, device=dev)
    if meta is None:
        meta = torch.empty(cm, dtype=torch.float32, device=dev)
    _expect(anchor, ca, torch.uint8, dev, "lynx_encode: anchor")
    _expect(residual, cr, torch.uint8, dev, "lynx_encode: residual")
    _expect(meta, cm, torch.float32, dev, "lynx_encode: meta")
    _check(lib().lynx_encode(_ptr(kv), B, L, H, D, page, C, alpha, _ptr(anchor), _ptr(residual),
                             _ptr(meta), _stream(dev)), "lynx_encode")
    return anchor, residual, meta


def _decode_out(anchor, L, out_dtype, out):
    B, NB, H, page, half = anchor.shape
    if out is None:
        out = torch.empty((B, L, H, half * 2), dtype=out_dtype, device=anchor.device)
    if out.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("lynx decode: output must be bfloat16 or float32")
    _expect(out, (B, L, H, half * 2), out.dtype, anchor.device, "lynx decode: out")
    code = LYNX_OUT_BF16 if out.dtype == torch.bfloat16 else LYNX_OUT_FP32
    return out, code, B, H, page, half * 2


def _check_decode_streams(what, anchor, residual, meta, L, page, C):
    if anchor.dim() != 5 or anchor.dtype != torch.uint8:
        raise ValueError(f"{what}: anchor must be uint8 [B][L/page][H_kv][page][D/2]")
    B, _, H, _, half = anchor.shape
    ca, cr, cm = stream_shapes(B, L, H, half * 2, page, C)
    _expect(anchor, ca, torch.uint8, anchor.device, f"{what}: anchor")
    if residual is not None:
        _expect(residual, cr, torch.uint8, anchor.device, f"{what}: residual")
    _expect(meta, cm, torch.float32, anchor.device, f"{what}: meta")


def lynx_decode_anchor(anchor, meta, L: int, page: int, C: int, alpha: float,
                       out_dtype=torch.bfloat16, out=None):
    """Anchor-only reconstruction -> out[B][L][H_kv][D]."""
    _need_cuda(anchor, meta, out)
    _check_decode_streams("lynx_decode_anchor", anchor, None, meta, L, page, C)
    out, code, B, H, P, D = _decode_out(anchor, L, out_dtype, out)
    _check(lib().lynx_decode_anchor(_ptr(anchor), _ptr(meta), B, L, H, D, page, C, alpha,
                                    _ptr(out), code, _stream(anchor.device)),
           "lynx_decode_anchor")
    return out


def lynx_decode_full(anchor, residual, meta, L: int, page: int, C: int, alpha: float,
                     out_dtype=torch.bfloat16, out=None):
    """Anchor + Residual reconstruction -> out[B][L][H_kv][D]."""
    _need_cuda(anchor, residual, meta, out)
    _check_decode_streams("lynx_decode_full", anchor, residual, meta, L, page, C)
    if residual is None:
        raise ValueError("lynx_decode_full: residual is required")
    out, code, B, H, P, D = _decode_out(anchor, L, out_dtype, out)
    _check(lib().lynx_decode_full(_ptr(anchor), _ptr(residual), _ptr(meta), B, L, H, D, page, C,
                                  alpha, _ptr(out), code, _stream(anchor.device)),
           "lynx_decode_full")
    return out


# ----------------------------------------------------------------- paged

def paged_pool_shapes(num_blocks: int, H_kv: int, D: int, page: int, C: int):
    """Tensor shapes of the (anchor, residual, meta) pools of num_blocks pages."""
    codes = (num_blocks, H_kv, page, D // 2)
    return codes, codes, (num_blocks, H_kv, 2 + 2 * (page // C), D)


def _check_table(block_table, B, NB):
    if block_table.dtype != torch.int32 or tuple(block_table.shape) != (B, NB):
        raise ValueError(f"block_table must be int32 [{B}][{NB}]")


def lynx_encode_paged(kv: torch.Tensor, page: int, C: int, alpha: float, block_table,
                      num_blocks: int, anchor_pool=None, residual_pool=None, meta_pool=None):
    """lynx_encode into pools of num_blocks pages through block_table [B][L/page]
    (int32).  Returns (anchor_pool, residual_pool, meta_pool)."""
    _need_cuda(kv, block_table, anchor_pool, residual_pool, meta_pool)
    if kv.dtype != torch.bfloat16 or kv.dim() != 4:
        raise ValueError("lynx_encode_paged: kv must be a 4-D bfloat16 tensor")
    B, L, H, D = kv.shape
    _check_table(block_table, B, L // page)
    ca, cr, cm = paged_pool_shapes(num_blocks, H, D, page, C)
    dev = kv.device
    if anchor_pool is None:
        anchor_pool = torch.empty(ca, dtype=torch.uint8, device=dev)
    if residual_pool is None:
        residual_pool = torch.empty(cr, dtype=torch.uint8, device=dev)
    if meta_pool is None:
        meta_pool = torch.empty(cm, dtype=torch.float32, device=dev)
    _expect(anchor_pool, ca, torch.uint8, dev, "lynx_encode_paged: anchor pool")
    _expect(residual_pool, cr, torch.uint8, dev, "lynx_encode_paged: residual pool")
    _expect(meta_pool, cm, torch.float32, dev, "lynx_encode_paged: meta pool")
    _check(lib().lynx_encode_paged(_ptr(kv), B, L, H, D, page, C, alpha, _ptr(block_table),
                                   num_blocks, _ptr(anchor_pool), _ptr(residual_pool),
                                   _ptr(meta_pool), _stream(dev)), "lynx_encode_paged")
    return anchor_pool, residual_pool, meta_pool


def lynx_decode_paged(anchor_pool, residual_pool, meta_pool, block_table, L: int, page: int,
                      C: int, alpha: float, mode: int, out_dtype=torch.bfloat16, out=None):
    """Decode paged streams (mode LYNX_ANCHOR or LYNX_FULL) -> out[B][L][H_kv][D]."""
    _need_cuda(anchor_pool, residual_pool, meta_pool, block_table, out)
    num_blocks, H, P, half = anchor_pool.shape
    B = block_table.shape[0]
    _check_table(block_table, B, L // page)
    if out is None:
        out = torch.empty((B, L, H, half * 2), dtype=out_dtype, device=anchor_pool.device)
    if out.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("lynx decode: output must be bfloat16 or float32")
    dev = anchor_pool.device
    shapes = paged_pool_shapes(num_blocks, H, half * 2, page, C)
    _expect(anchor_pool, shapes[0], torch.uint8, dev, "lynx_decode_paged: anchor pool")
    if mode == LYNX_FULL:
        _expect(residual_pool, shapes[1], torch.uint8, dev, "lynx_decode_paged: residual pool")
    _expect(meta_pool, shapes[2], torch.float32, dev, "lynx_decode_paged: meta pool")
    _expect(out, (B, L, H, half * 2), out.dtype, dev, "lynx_decode_paged: out")
    code = LYNX_OUT_BF16 if out.dtype == torch.bfloat16 else LYNX_OUT_FP32
    _check(lib().lynx_decode_paged(_ptr(anchor_pool), _ptr(residual_pool), _ptr(meta_pool),
                                   _ptr(block_table), num_blocks, B, L, H, half * 2, page, C,
                                   alpha, mode, _ptr(out), code, _stream(anchor_pool.device)),
           "lynx_decode_paged")
    return out


def lynx_spec_verify(p, q, draft_tokens, u, r, n_accepted=None, next_token=None):
    """Eq. 10-11 for a batch: p [batch][T+1][V] f32, q [batch][T][V] f32,
    draft_tokens [batch][T] int32, u [batch][T] f32, r [batch] int32 holding
    uint32 bits.  Returns (n_accepted, next_token), int32 [batch]."""
    _need_cuda(p, q, draft_tokens, u, r, n_accepted, next_token)
    batch, T1, V = p.shape
    T = T1 - 1
    if p.dtype != torch.float32 or q.dtype != torch.float32 or u.dtype != torch.float32:
        raise ValueError("lynx_spec_verify: p, q and u must be float32")
    if draft_tokens.dtype != torch.int32 or r.dtype != torch.int32:
        raise ValueError("lynx_spec_verify: draft_tokens and r must be int32 tensors")
    if tuple(q.shape) != (batch, T, V) or tuple(draft_tokens.shape) != (batch, T) or \
            tuple(u.shape) != (batch, T) or tuple(r.shape) != (batch,):
        raise ValueError("lynx_spec_verify: shapes")
    if n_accepted is None:
        n_accepted = torch.empty(batch, dtype=torch.int32, device=p.device)
    if next_token is None:
        next_token = torch.empty(batch, dtype=torch.int32, device=p.device)
    _check(lib().lynx_spec_verify(_ptr(p), _ptr(q), _ptr(draft_tokens), _ptr(u), _ptr(r), batch,
                                  T, V, _ptr(n_accepted), _ptr(next_token), _stream(p.device)),
           "lynx_spec_verify")
    return n_accepted, next_token


def lynx_wait_selftest(limit_ns: int, arrive, device) -> int:
    """Run the bounded-wait check; returns 1 (barrier completed) or 2 (the
    wait gave up after limit_ns); with arrive == 2 the verification pass's
    wait and abort word: 3 (both waits ended as they must) or 4."""
    st = torch.zeros(1, dtype=torch.int32, device=device)
    _check(lib().lynx_wait_selftest(limit_ns, int(arrive), _ptr(st), _stream(st.device)),
           "lynx_wait_selftest")
    return int(st.item())


def lynx_device_errors() -> int:
    bits = ctypes.c_uint()
    _check(lib().lynx_device_errors(ctypes.byref(bits)), "lynx_device_errors")
    return bits.value


# ------------------------------------------------------- split-stream transfer

LYNX_OP_ENCODE, LYNX_OP_COPY_ANCHOR, LYNX_OP_COPY_META, LYNX_OP_COPY_RESIDUAL = 0, 1, 2, 3
LYNX_OP_DECODE_ANCHOR, LYNX_OP_UPGRADE, LYNX_OP_NONE = 4, 5, -1
LYNX_Q_COPY, LYNX_Q_HI, LYNX_Q_LO = 0, 1, 2


class SplitOp(ctypes.Structure):
    """lynx_split_op of include/lynx.h."""
    _fields_ = [("kind", ctypes.c_int32), ("queue", ctypes.c_int32), ("group", ctypes.c_int64),
                ("page0", ctypes.c_int64), ("n_pages", ctypes.c_int64),
                ("offset", ctypes.c_int64), ("bytes", ctypes.c_int64),
                ("wait_kind", ctypes.c_int32 * 2), ("wait_group", ctypes.c_int64 * 2)]


class LynxHeader(ctypes.Structure):
    """lynx_header of include/lynx.h (128 bytes)."""
    _fields_ = [("magic", ctypes.c_char * 8), ("version", ctypes.c_uint32),
                ("header_bytes", ctypes.c_uint32), ("B", ctypes.c_int64), ("L", ctypes.c_int64),
                ("H_kv", ctypes.c_int32), ("D", ctypes.c_int32), ("page", ctypes.c_int32),
                ("C", ctypes.c_int32), ("alpha", ctypes.c_float), ("flags", ctypes.c_uint32),
                ("anchor_offset", ctypes.c_uint64), ("anchor_bytes", ctypes.c_uint64),
                ("meta_offset", ctypes.c_uint64), ("meta_bytes", ctypes.c_uint64),
                ("residual_offset", ctypes.c_uint64), ("residual_bytes", ctypes.c_uint64),
                ("total_bytes", ctypes.c_uint64), ("reserved", ctypes.c_uint32 * 3),
                ("header_crc", ctypes.c_uint32)]


def lynx_split_plan(B: int, L: int, H_kv: int, D: int, page: int, C: int, pages_per_group: int,
                    send: bool = False, with_decode: bool = True):
    """The transfer schedule as a list of dicts, in issue order."""
    n = ctypes.c_int64()
    rc = lib().lynx_split_plan(B, L, H_kv, D, page, C, pages_per_group, int(send),
                               int(with_decode), None, 0, ctypes.byref(n))
    if rc not in (LYNX_OK, LYNX_EWORKSPACE):
        _check(rc, "lynx_split_plan")
    buf = (SplitOp * max(1, n.value))()
    _check(lib().lynx_split_plan(B, L, H_kv, D, page, C, pages_per_group, int(send),
                                 int(with_decode), buf, n.value, ctypes.byref(n)),
           "lynx_split_plan")
    return [{"kind": o.kind, "queue": o.queue, "group": o.group, "page0": o.page0,
             "n_pages": o.n_pages, "offset": o.offset, "bytes": o.bytes,
             "waits": [(o.wait_kind[i], o.wait_group[i]) for i in range(2)
                       if o.wait_kind[i] != LYNX_OP_NONE]} for o in buf[:n.value]]


def _need_host(*ts):
    for t in ts:
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("lynx: host buffers must be contiguous CPU tensors (pinned)")


def _raw_stream(s):
    return ctypes.c_void_p(s.cuda_stream) if s is not None else None


def _raw_event(ev, stream):
    """Handle of a torch.cuda.Event, created (by a first record) if still lazy."""
    if ev is None:
        return None
    if not ev.cuda_event:
        ev.record(stream if stream is not None else torch.cuda.current_stream())
    return ctypes.c_void_p(ev.cuda_event)


def lynx_split_receive(host, dev, L: int, page: int, C: int, alpha: float, pages_per_group: int,
                       out=None, copy_stream=None, hi_stream=None, lo_stream=None,
                       anchor_ready=None, full_ready=None):
    """Receiver side: host = (anchor, residual, meta) CPU tensors, dev = the
    same three CUDA tensors (stream_shapes); out (optional) is decoded from
    the Anchor as it lands and upgraded in place to the full decode."""
    ha, hr, hm = host
    da, dr, dm = dev
    _need_host(ha, hr, hm)
    _need_cuda(da, dr, dm, out)
    B, NB, H, P, half = da.shape
    code = LYNX_OUT_BF16
    if out is not None:
        if out.dtype not in (torch.bfloat16, torch.float32):
            raise ValueError("lynx_split_receive: out must be bfloat16 or float32")
        code = LYNX_OUT_BF16 if out.dtype == torch.bfloat16 else LYNX_OUT_FP32
    _check(lib().lynx_split_receive(_ptr(ha), _ptr(hm), _ptr(hr), _ptr(da), _ptr(dm), _ptr(dr),
                                    B, L, H, half * 2, page, C, alpha, pages_per_group, _ptr(out),
                                    code, _raw_stream(copy_stream), _raw_stream(hi_stream),
                                    _raw_stream(lo_stream), _raw_event(anchor_ready, hi_stream),
                                    _raw_event(full_ready, lo_stream)),
           "lynx_split_receive")


def lynx_split_send(kv, page: int, C: int, alpha: float, dev, host, pages_per_group: int,
                    hi_stream=None, copy_stream=None, anchor_sent=None, all_sent=None):
    """Sender side: encode kv into dev = (anchor, residual, meta) group by
    group and copy each group to host = (anchor, residual, meta) CPU tensors,
    every Residual after the last Anchor."""
    da, dr, dm = dev
    ha, hr, hm = host
    _need_cuda(kv, da, dr, dm)
    _need_host(ha, hr, hm)
    B, L, H, D = kv.shape
    _check(lib().lynx_split_send(_ptr(kv), B, L, H, D, page, C, alpha, _ptr(da), _ptr(dm),
                                 _ptr(dr), _ptr(ha), _ptr(hm), _ptr(hr), pages_per_group,
                                 _raw_stream(hi_stream), _raw_stream(copy_stream),
                                 _raw_event(anchor_sent, copy_stream),
                                 _raw_event(all_sent, copy_stream)),
           "lynx_split_send")


def lynx_header_init(B: int, L: int, H_kv: int, D: int, page: int, C: int, alpha: float,
                     with_residual: bool = True) -> bytes:
    """The 128-byte header of a serialized request."""
    h = LynxHeader()
    _check(lib().lynx_header_init(ctypes.byref(h), B, L, H_kv, D, page, C, alpha,
                                  int(with_residual)), "lynx_header_init")
    return bytes(h)


def lynx_header_check(buf: bytes) -> LynxHeader:
    """Validate a header; returns it parsed, or raises LynxError."""
    if len(buf) < ctypes.sizeof(LynxHeader):
        raise ValueError("lynx_header_check: fewer than 128 bytes")
    h = LynxHeader.from_buffer_copy(bytes(buf[:ctypes.sizeof(LynxHeader)]))
    _check(lib().lynx_header_check(ctypes.byref(h)), "lynx_header_check")
    return h


# ------------------------------------------------------- comparison points

def lynx_int_encode(kv, bits: int, codes=None, meta=None):
    """Linear INT-`bits` baseline (Eq. 4) of kv[..][128] BF16: one scale and
    zero point per row of 128 channels.  Returns (codes, meta)."""
    _need_cuda(kv, codes, meta)
    if kv.dtype != torch.bfloat16 or kv.shape[-1] != 128:
        raise ValueError("lynx_int_encode: kv must be bfloat16 with 128 channels")
    rows = kv.numel() // 128
    if codes is None:
        codes = torch.empty(kv.shape[:-1] + (128 * bits // 8,), dtype=torch.uint8,
                            device=kv.device)
    if meta is None:
        meta = torch.empty(kv.shape[:-1] + (2,), dtype=torch.float32, device=kv.device)
    _check(lib().lynx_int_encode(_ptr(kv), rows, 128, bits, _ptr(codes), _ptr(meta),
                                 _stream(kv.device)), "lynx_int_encode")
    return codes, meta


def lynx_int_decode(codes, meta, bits: int, out_dtype=torch.bfloat16, out=None):
    _need_cuda(codes, meta, out)
    rows = meta.numel() // 2
    if out is None:
        out = torch.empty(meta.shape[:-1] + (128,), dtype=out_dtype, device=codes.device)
    code = LYNX_OUT_BF16 if out.dtype == torch.bfloat16 else LYNX_OUT_FP32
    _check(lib().lynx_int_decode(_ptr(codes), _ptr(meta), rows, 128, bits, _ptr(out), code,
                                 _stream(codes.device)), "lynx_int_decode")
    return out


def lynx_split_bits(anchor, residual, k: int, anchor_k=None, residual_k=None):
    """Re-split 4+4 streams [B][NB][H][P][64] into a k + (8-k) split:
    returns (anchor_k [B][NB][H][P][16k], residual_k [..][16(8-k)])."""
    _need_cuda(anchor, residual, anchor_k, residual_k)
    shp = anchor.shape[:-1]
    rows = anchor.numel() // 64
    if anchor_k is None:
        anchor_k = torch.empty(shp + (16 * k,), dtype=torch.uint8, device=anchor.device)
    if residual_k is None:
        residual_k = torch.empty(shp + (16 * (8 - k),), dtype=torch.uint8, device=anchor.device)
    _check(lib().lynx_split_bits(_ptr(anchor), _ptr(residual), rows, 128, k, _ptr(anchor_k),
                                 _ptr(residual_k), _stream(anchor.device)), "lynx_split_bits")
    return anchor_k, residual_k


def lynx_join_bits(anchor_k, residual_k, k: int, anchor=None, residual=None):
    _need_cuda(anchor_k, residual_k, anchor, residual)
    shp = anchor_k.shape[:-1]
    rows = anchor_k.numel() // (16 * k)
    if anchor is None:
        anchor = torch.empty(shp + (64,), dtype=torch.uint8, device=anchor_k.device)
    if residual is None:
        residual = torch.empty(shp + (64,), dtype=torch.uint8, device=anchor_k.device)
    _check(lib().lynx_join_bits(_ptr(anchor_k), _ptr(residual_k), rows, 128, k, _ptr(anchor),
                                _ptr(residual), _stream(anchor_k.device)), "lynx_join_bits")
    return anchor, residual


def lynx_decode_anchor_bits(anchor_k, meta, L: int, page: int, C: int, alpha: float, k: int,
                            out_dtype=torch.bfloat16, out=None):
    """Anchor-only decode of a k-bit Anchor stream [B][NB][H][P][16k]."""
    _need_cuda(anchor_k, meta, out)
    B, NB, H = anchor_k.shape[:3]
    if out is None:
        out = torch.empty((B, L, H, 128), dtype=out_dtype, device=anchor_k.device)
    code = LYNX_OUT_BF16 if out.dtype == torch.bfloat16 else LYNX_OUT_FP32
    _check(lib().lynx_decode_anchor_bits(_ptr(anchor_k), _ptr(meta), B, L, H, 128, page, C, alpha,
                                         k, _ptr(out), code, _stream(anchor_k.device)),
           "lynx_decode_anchor_bits")
    return out


def lynx_a1_encode(kv, page: int, alpha: float = 100.0):
    """The Appendix A.1 variant of kv[B][L][H][128] BF16: returns (anchor,
    residual, meta[B][L/page][H][1 + page/16][128])."""
    _need_cuda(kv)
    if kv.dtype != torch.bfloat16 or kv.dim() != 4:
        raise ValueError("lynx_a1_encode: kv must be a 4-D bfloat16 tensor")
    B, L, H, D = kv.shape
    codes = (B, L // page, H, page, D // 2)
    anchor = torch.empty(codes, dtype=torch.uint8, device=kv.device)
    residual = torch.empty(codes, dtype=torch.uint8, device=kv.device)
    meta = torch.empty((B, L // page, H, 1 + page // 16, D), dtype=torch.float32,
                       device=kv.device)
    _check(lib().lynx_a1_encode(_ptr(kv), B, L, H, D, page, alpha, _ptr(anchor), _ptr(residual),
                                _ptr(meta), _stream(kv.device)), "lynx_a1_encode")
    return anchor, residual, meta


def lynx_a1_decode(anchor, residual, meta, L: int, page: int, alpha: float = 100.0,
                   out_dtype=torch.bfloat16, out=None):
    """Decode of the A.1 variant; residual None gives the Anchor-only decode."""
    _need_cuda(anchor, residual, meta, out)
    B, NB, H, P, half = anchor.shape
    if out is None:
        out = torch.empty((B, L, H, half * 2), dtype=out_dtype, device=anchor.device)
    code = LYNX_OUT_BF16 if out.dtype == torch.bfloat16 else LYNX_OUT_FP32
    _check(lib().lynx_a1_decode(_ptr(anchor), _ptr(residual), _ptr(meta), B, L, H, half * 2, page,
                                alpha, _ptr(out), code, _stream(anchor.device)),
           "lynx_a1_decode")
    return out


# ----------------------------------------------------------------- attention

def lynx_attn_workspace_bytes(batch: int, T: int, H_q: int, L: int, H_kv: int, D: int,
                              page: int) -> int:
    n = ctypes.c_size_t()
    _check(lib().lynx_attn_workspace_bytes(batch, T, H_q, L, H_kv, D, page, ctypes.byref(n)),
           "lynx_attn_workspace_bytes")
    return n.value


def _check_attn_io(what, q, ks, vs, L, page, C, mode, out, workspace, need, pools=False):
    """Shapes, types and devices of everything an attention call reads or
    writes: q [batch][T][H_q][D] bf16; K and V streams of one layout (dense
    [batch][L/page][H_kv][...], or pools [num_blocks][H_kv][...]); residuals
    present in full mode; out [batch][T][H_q][D] float32; a workspace of at
    least `need` bytes."""
    batch, T, H_q, D = q.shape
    dev = q.device
    for name, (a, r, m) in (("k", ks), ("v", vs)):
        if a.dtype != torch.uint8 or a.dim() != (4 if pools else 5):
            raise ValueError(f"{what}: {name} anchor must be uint8 "
                             + ("[num_blocks][H_kv][page][D/2]" if pools
                                else "[batch][L/page][H_kv][page][D/2]"))
        if pools:
            nb, H_kv = a.shape[0], a.shape[1]
            codes = (nb, H_kv, page, D // 2)
            mshape = (nb, H_kv, 2 + 2 * (page // C), D)
        else:
            H_kv = a.shape[2]
            codes, _, mshape = stream_shapes(batch, L, H_kv, D, page, C)
        _expect(a, codes, torch.uint8, dev, f"{what}: {name} anchor")
        if mode == LYNX_FULL:
            _expect(r, codes, torch.uint8, dev, f"{what}: {name} residual")
        _expect(m, mshape, torch.float32, dev, f"{what}: {name} meta")
    if tuple(ks[0].shape) != tuple(vs[0].shape):
        raise ValueError(f"{what}: K and V streams differ in shape")
    _expect(out, (batch, T, H_q, D), torch.float32, dev, f"{what}: out")
    if workspace is not None:
        if workspace.device != dev:
            raise ValueError(f"{what}: workspace on {workspace.device}, expected {dev}")
        if workspace.numel() * workspace.element_size() < need:
            raise ValueError(f"{what}: workspace holds "
                             f"{workspace.numel() * workspace.element_size()} bytes, "
                             f"the call needs {need}")


def lynx_attn_decode(q, k_streams, v_streams, L: int, page: int, C: int, alpha: float,
                     mode: int, out=None, workspace=None, k_tail=None, v_tail=None):
    """q[batch][T][H_q][D] bf16; k_streams / v_streams = (anchor, residual or
    None, meta) from lynx_encode of K and V.  With k_tail / v_tail
    ([batch][T][H_kv][D] bf16, the draft tokens' own keys and values) query
    token t also attends to draft tokens 0..t (lynx_attn_decode_tail).
    Returns out[batch][T][H_q][D] f32."""
    ka, kr, km = k_streams
    va, vr, vm = v_streams
    _need_cuda(q, ka, kr, km, va, vr, vm, out, workspace, k_tail, v_tail)
    if (k_tail is None) != (v_tail is None):
        raise ValueError("lynx_attn_decode: give both k_tail and v_tail, or neither")
    if q.dtype != torch.bfloat16 or q.dim() != 4:
        raise ValueError("lynx_attn_decode: q must be a 4-D bfloat16 tensor")
    batch, T, H_q, D = q.shape
    if ka.dim() != 5:
        raise ValueError("lynx_attn_decode: streams must be [batch][L/page][H_kv][...]")
    H_kv = ka.shape[2]
    if out is None:
        out = torch.empty((batch, T, H_q, D), dtype=torch.float32, device=q.device)
    need = lynx_attn_workspace_bytes(batch, T, H_q, L, H_kv, D, page)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check_attn_io("lynx_attn_decode", q, k_streams, v_streams, L, page, C, mode, out,
                   workspace, need)
    if k_tail is not None:
        for t in (k_tail, v_tail):
            if t.dtype != torch.bfloat16 or tuple(t.shape) != (batch, T, H_kv, D) or \
                    not t.is_contiguous():
                raise ValueError("lynx_attn_decode: tails must be contiguous bfloat16 "
                                 "[batch][T][H_kv][D]")
        _check(lib().lynx_attn_decode_tail(_ptr(q), batch, T, H_q, _ptr(ka), _ptr(kr),
                                           _ptr(km), _ptr(va), _ptr(vr), _ptr(vm), L, H_kv, D,
                                           page, C, alpha, mode, _ptr(k_tail), _ptr(v_tail),
                                           _ptr(out), _ptr(workspace),
                                           workspace.numel() * workspace.element_size(),
                                           _stream(q.device)), "lynx_attn_decode_tail")
        return out
    _check(lib().lynx_attn_decode(_ptr(q), batch, T, H_q, _ptr(ka), _ptr(kr), _ptr(km),
                                  _ptr(va), _ptr(vr), _ptr(vm), L, H_kv, D, page, C, alpha,
                                  mode, _ptr(out), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(),
                                  _stream(q.device)), "lynx_attn_decode")
    return out


def lynx_attn_decode_tail(q, k_streams, v_streams, L: int, page: int, C: int, alpha: float,
                          mode: int, k_tail, v_tail, out=None, workspace=None):
    """lynx_attn_decode_tail: query token t attends to the L cached tokens and
    to the draft tokens 0..t given by k_tail / v_tail ([batch][T][H_kv][D] bf16)."""
    if k_tail is None or v_tail is None:
        raise ValueError("lynx_attn_decode_tail: k_tail and v_tail are required")
    return lynx_attn_decode(q, k_streams, v_streams, L, page, C, alpha, mode, out=out,
                            workspace=workspace, k_tail=k_tail, v_tail=v_tail)


def lynx_attn_decode_paged(q, k_pools, v_pools, block_table, L: int, page: int, C: int,
                           alpha: float, mode: int, out=None, workspace=None, k_tail=None,
                           v_tail=None):
    """lynx_attn_decode(_tail) over paged K and V pools (anchor, residual or None,
    meta) read through block_table [batch][L/page] (int32)."""
    ka, kr, km = k_pools
    va, vr, vm = v_pools
    _need_cuda(q, ka, kr, km, va, vr, vm, block_table, out, workspace, k_tail, v_tail)
    if (k_tail is None) != (v_tail is None):
        raise ValueError("lynx_attn_decode_paged: give both k_tail and v_tail, or neither")
    if q.dtype != torch.bfloat16 or q.dim() != 4:
        raise ValueError("lynx_attn_decode_paged: q must be a 4-D bfloat16 tensor")
    batch, T, H_q, D = q.shape
    if ka.dim() != 4:
        raise ValueError("lynx_attn_decode_paged: pools must be [num_blocks][H_kv][...]")
    num_blocks, H_kv = ka.shape[0], ka.shape[1]
    _check_table(block_table, batch, L // page)
    if out is None:
        out = torch.empty((batch, T, H_q, D), dtype=torch.float32, device=q.device)
    need = lynx_attn_workspace_bytes(batch, T, H_q, L, H_kv, D, page)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check_attn_io("lynx_attn_decode_paged", q, k_pools, v_pools, L, page, C, mode, out,
                   workspace, need, pools=True)
    if k_tail is not None:
        for t in (k_tail, v_tail):
            _expect(t, (batch, T, H_kv, D), torch.bfloat16, q.device,
                    "lynx_attn_decode_paged: tail")
    _check(lib().lynx_attn_decode_paged(_ptr(q), batch, T, H_q, _ptr(ka), _ptr(kr), _ptr(km),
                                        _ptr(va), _ptr(vr), _ptr(vm), _ptr(block_table),
                                        num_blocks, L, H_kv, D, page, C, alpha, mode,
                                        _ptr(k_tail), _ptr(v_tail), _ptr(out), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(),
                                        _stream(q.device)),
           "lynx_attn_decode_paged")
    return out


def lynx_attn_decode_noalloc(q, k_streams, v_streams, L: int, page: int, C: int,
                             alpha: float, mode: int, out=None):
    """lynx_attn_decode with the library's built-in scratch instead of a
    workspace (for callers that cannot allocate device memory).  `out` must
    be given by such callers; if it is None it is allocated here for
    convenience."""
    ka, kr, km = k_streams
    va, vr, vm = v_streams
    _need_cuda(q, ka, kr, km, va, vr, vm, out)
    if q.dtype != torch.bfloat16 or q.dim() != 4:
        raise ValueError("lynx_attn_decode_noalloc: q must be a 4-D bfloat16 tensor")
    batch, T, H_q, D = q.shape
    if ka.dim() != 5:
        raise ValueError("lynx_attn_decode_noalloc: streams must be [batch][L/page][H_kv][...]")
    H_kv = ka.shape[2]
    if out is None:
        out = torch.empty((batch, T, H_q, D), dtype=torch.float32, device=q.device)
    _check_attn_io("lynx_attn_decode_noalloc", q, k_streams, v_streams, L, page, C, mode, out,
                   None, 0)
    _check(lib().lynx_attn_decode_noalloc(_ptr(q), batch, T, H_q, _ptr(ka), _ptr(kr), _ptr(km),
                                          _ptr(va), _ptr(vr), _ptr(vm), L, H_kv, D, page, C,
                                          alpha, mode, _ptr(out), _stream(q.device)),
           "lynx_attn_decode_noalloc")
    return out


# ----------------------------------------------------------------- tables

def lynx_compander_thresholds(alpha: float):
    buf = (ctypes.c_float * 127)()
    _check(lib().lynx_compander_thresholds(alpha, ctypes.cast(buf, ctypes.c_void_p)),
           "lynx_compander_thresholds")
    return list(buf)


def lynx_expand_table(alpha: float):
    buf = (ctypes.c_float * 128)()
    _check(lib().lynx_expand_table(alpha, ctypes.cast(buf, ctypes.c_void_p)),
           "lynx_expand_table")
    return list(buf)


def lynx_compander_selfcheck(alpha: float, device="cuda"):
    """[values checked, wrong unflagged, flagged, max |error| in 2^-32 of Y]."""
    counts = torch.zeros(4, dtype=torch.int64, device=device)
    _check(lib().lynx_compander_selfcheck(alpha, _ptr(counts), _stream(counts.device)),
           "lynx_compander_selfcheck")
    return [int(v) for v in counts.cpu().tolist()]


def lynx_wait_timeouts() -> int:
    flag = ctypes.c_uint()
    _check(lib().lynx_wait_timeouts(ctypes.byref(flag)), "lynx_wait_timeouts")
    return flag.value


def lynx_status_string(code: int) -> str:
    return lib().lynx_status_string(code).decode()


def lynx_last_error() -> str:
    return lib().lynx_last_error().decode(errors="replace")
