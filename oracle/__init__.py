"""CPU oracle for the MXFP4 latent-MoE layer -- TEST INFRASTRUCTURE ONLY.

Only tests/, the smoke check in __graft_entry__ and the CPU-baseline leg of
bench.py may import this package. The CUDA product path never does.

Thin ctypes wrapper over libmoe_oracle.so (built by oracle/build.py); numpy
arrays in, numpy arrays out. Each function's arithmetic lives in
moe_oracle.cpp, whose header cites the page sections it restates.
"""
import ctypes
import os

import numpy as np

from .build import LIB, build_oracle

_lib = None

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            build_oracle()
        L = ctypes.CDLL(LIB)
        sig = {
            "orc_e2m1_value": (ctypes.c_double, [ctypes.c_uint8]),
            "orc_e4m3_value": (ctypes.c_double, [ctypes.c_uint8]),
            "orc_e8m0_value": (ctypes.c_double, [ctypes.c_uint8]),
            "orc_e4m3_encode_rne_sat": (ctypes.c_uint8, [ctypes.c_double]),
            "orc_mx_quant_block": (None, [_f32p, _u8p, _u8p]),
            "orc_mx_quant_rows": (None, [_f32p, _i64, _i64, _u8p, _u8p]),
            "orc_mx_quant_rows_bf16": (None, [_u16p, _i64, _i64, _u8p, _u8p]),
            "orc_route_topk": (None, [_f32p, _i64, _i32, _i32, _i32p, _f32p]),
            "orc_permute": (_i32, [_i32p, _i64, _i32, _i32, _i32, _i32p, _i32p, _i32p, _i32p, _i64]),
            "orc_expert_stage1": (None, [_u8p, _u8p, _i32, _i32, _u8p, _u8p, _f64p]),
            "orc_expert_stage2": (None, [_u8p, _u8p, _i32, _i32, _u8p, _u8p, _f64p]),
            "orc_bf16_rne": (ctypes.c_uint16, [ctypes.c_double]),
            "orc_moe_forward": (None, [_u16p, _f32p, _i64, _i32, _i32, _i32, _i32,
                                       _u8p, _u8p, _u8p, _u8p, _u16p, _i32p, _f32p, _f64p, _i32]),
            "orc_expert_bytes": (_i64, [_i32, _i32]),
            "orc_e2m1_encode_rne_sat": (ctypes.c_uint8, [ctypes.c_double]),
            "orc_gemm_bf16": (None, [_u16p, _u16p, _i64, _i64, _i64, _f64p]),
            "orc_bf16_rne_n": (None, [_f64p, _i64, _u16p]),
            "orc_gemm_bf16_swiglu": (None, [_u16p, _u16p, _i64, _i64, _i64, _f64p]),
            "orc_mxfp4_quant_block": (None, [_f32p, _u8p, _u8p]),
            "orc_mxfp4_quant_rows": (None, [_f32p, _i64, _i64, _u8p, _u8p]),
            "orc_mxfp4_quant_rows_bf16": (None, [_u16p, _i64, _i64, _u8p, _u8p]),
            "orc_expert_stage1_a4": (None, [_u8p, _u8p, _i32, _i32, _u8p, _u8p, _f64p]),
            "orc_moe_forward_a4w4": (None, [_u16p, _f32p, _i64, _i32, _i32, _i32, _i32,
                                            _u8p, _u8p, _u8p, _u8p, _u16p, _i32p, _f32p,
                                            _f64p, _i32]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _p(a, ptype):
    if a is None:
        return ctypes.cast(None, ptype)
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ptype)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def e2m1_value(code):
    return lib().orc_e2m1_value(int(code))


def e4m3_value(code):
    return lib().orc_e4m3_value(int(code))


def e8m0_value(code):
    return lib().orc_e8m0_value(int(code))


def e4m3_encode(v):
    return lib().orc_e4m3_encode_rne_sat(float(v))


def bf16_rne(v):
    return lib().orc_bf16_rne(float(v))


def mx_quant_rows(v):
    """fp32 [rows][K] -> (codes u8 [rows][K], scales u8 [rows][K/32])."""
    v = _c(v, np.float32)
    rows, K = v.shape
    codes = np.empty((rows, K), np.uint8)
    scales = np.empty((rows, K // 32), np.uint8)
    lib().orc_mx_quant_rows(_p(v, _f32p), rows, K, _p(codes, _u8p), _p(scales, _u8p))
    return codes, scales


def mx_quant_rows_bf16(x_bits):
    """bf16 bit patterns (uint16) [rows][K] -> (codes, scales)."""
    x = _c(x_bits, np.uint16)
    rows, K = x.shape
    codes = np.empty((rows, K), np.uint8)
    scales = np.empty((rows, K // 32), np.uint8)
    lib().orc_mx_quant_rows_bf16(_p(x, _u16p), rows, K, _p(codes, _u8p), _p(scales, _u8p))
    return codes, scales


def e2m1_encode(v):
    return lib().orc_e2m1_encode_rne_sat(float(v))


def mxfp4_quant_rows(v):
    """fp32 [rows][K] -> (packed E2M1 u8 [rows][K/2], scales u8 [rows][K/32])."""
    v = _c(v, np.float32)
    rows, K = v.shape
    packed = np.empty((rows, K // 2), np.uint8)
    scales = np.empty((rows, K // 32), np.uint8)
    lib().orc_mxfp4_quant_rows(_p(v, _f32p), rows, K, _p(packed, _u8p), _p(scales, _u8p))
    return packed, scales


def mxfp4_quant_rows_bf16(x_bits):
    """bf16 bit patterns (uint16) [rows][K] -> (packed E2M1 [rows][K/2], scales)."""
    x = _c(x_bits, np.uint16)
    rows, K = x.shape
    packed = np.empty((rows, K // 2), np.uint8)
    scales = np.empty((rows, K // 32), np.uint8)
    lib().orc_mxfp4_quant_rows_bf16(_p(x, _u16p), rows, K, _p(packed, _u8p), _p(scales, _u8p))
    return packed, scales


def route_topk(logits, k):
    lg = _c(logits, np.float32)
    T, E = lg.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    lib().orc_route_topk(_p(lg, _f32p), T, E, k, _p(ids, _i32p), _p(w, _f32p))
    return ids, w


def permute(ids, E, pad_m, rows_capacity=None):
    ids = _c(ids, np.int32)
    T, k = ids.shape
    if rows_capacity is None:
        rows_capacity = T * k + min(E, T * k) * (pad_m - 1)
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    slot_to_row = np.empty(T * k, np.int32)
    row_to_slot = np.full(max(rows_capacity, 1), -7, np.int32)
    rc = lib().orc_permute(_p(ids, _i32p), T, E, k, pad_m, _p(counts, _i32p), _p(offsets, _i32p),
                           _p(slot_to_row, _i32p), _p(row_to_slot, _i32p), rows_capacity)
    if rc != 0:
        raise ValueError("oracle permute rejected its input")
    return dict(counts=counts, offsets=offsets, slot_to_row=slot_to_row,
                row_to_slot=row_to_slot[: int(offsets[E])])


def expert_stage1(xq, xs, w13_e, w13s_e):
    xq, xs = _c(xq, np.uint8), _c(xs, np.uint8)
    w13_e, w13s_e = _c(w13_e, np.uint8), _c(w13s_e, np.uint8)
    d = xq.shape[0]
    I = w13_e.shape[0] // 2
    h = np.empty(I, np.float64)
    lib().orc_expert_stage1(_p(xq, _u8p), _p(xs, _u8p), d, I, _p(w13_e, _u8p),
                            _p(w13s_e, _u8p), _p(h, _f64p))
    return h


def expert_stage1_a4(xq, xs, w13_e, w13s_e):
    """Stage 1 with an MXFP4 activation row: xq packed E2M1 [d/2], xs [d/32]."""
    xq, xs = _c(xq, np.uint8), _c(xs, np.uint8)
    w13_e, w13s_e = _c(w13_e, np.uint8), _c(w13s_e, np.uint8)
    d = xq.shape[0] * 2
    I = w13_e.shape[0] // 2
    h = np.empty(I, np.float64)
    lib().orc_expert_stage1_a4(_p(xq, _u8p), _p(xs, _u8p), d, I, _p(w13_e, _u8p),
                               _p(w13s_e, _u8p), _p(h, _f64p))
    return h


def expert_stage2(hq, hs, w2_e, w2s_e):
    hq, hs = _c(hq, np.uint8), _c(hs, np.uint8)
    w2_e, w2s_e = _c(w2_e, np.uint8), _c(w2s_e, np.uint8)
    I = hq.shape[0]
    d = w2_e.shape[0]
    y = np.empty(d, np.float64)
    lib().orc_expert_stage2(_p(hq, _u8p), _p(hs, _u8p), I, d, _p(w2_e, _u8p),
                            _p(w2s_e, _u8p), _p(y, _f64p))
    return y


def moe_forward(x_bits, logits, k, w13, w13s, w2, w2s, threads=0, want_y64=False,
                a4w4=False):
    """Whole layer for independent tokens. x_bits bf16 patterns [n][d].
    a4w4: MXFP4 stage-1 activations (orc_moe_forward_a4w4).

    Returns dict(y=bf16 bits [n][d], ids, w, y64 (or None)).
    """
    x = _c(x_bits, np.uint16)
    lg = _c(logits, np.float32)
    w13, w13s, w2, w2s = (_c(a, np.uint8) for a in (w13, w13s, w2, w2s))
    n, d = x.shape
    E = lg.shape[1]
    I = w13.shape[1] // 2
    y = np.empty((n, d), np.uint16)
    ids = np.empty((n, max(k, 1)), np.int32)
    w = np.empty((n, max(k, 1)), np.float32)
    y64 = np.empty((n, d), np.float64) if want_y64 else None
    fn = lib().orc_moe_forward_a4w4 if a4w4 else lib().orc_moe_forward
    fn(_p(x, _u16p), _p(lg, _f32p), n, d, E, k, I, _p(w13, _u8p), _p(w13s, _u8p),
       _p(w2, _u8p), _p(w2s, _u8p), _p(y, _u16p), _p(ids, _i32p), _p(w, _f32p), _p(y64, _f64p),
       threads)
    return dict(y=y, ids=ids[:, :k], w=w[:, :k], y64=y64)


def _by_rows(fn, a, n_out, threads):
    """fn(a_rows, out_rows) over row chunks of a on `threads` host threads
    (0 = all cores; the rows are independent and the library call releases
    the interpreter lock)."""
    import concurrent.futures as cf
    M = a.shape[0]
    out = np.empty((M, n_out), np.float64)
    n = threads if threads > 0 else (os.cpu_count() or 1)
    n = max(1, min(n, M))
    if n == 1:
        fn(a, out)
        return out
    parts = [p for p in np.array_split(np.arange(M), n) if len(p)]

    def run(p):
        o = np.empty((len(p), n_out), np.float64)
        fn(np.ascontiguousarray(a[p[0]:p[-1] + 1]), o)
        out[p[0]:p[-1] + 1] = o

    with cf.ThreadPoolExecutor(len(parts)) as ex:
        list(ex.map(run, parts))
    return out


def gemm_bf16(a_bits, b_bits, threads=1):
    """C = A . B^T in fp64; a_bits [M][K], b_bits [N][K] bf16 bit patterns."""
    a, b = _c(a_bits, np.uint16), _c(b_bits, np.uint16)
    K = a.shape[1]
    N = b.shape[0]

    def fn(ar, c):
        lib().orc_gemm_bf16(_p(ar, _u16p), _p(b, _u16p), ar.shape[0], N, K, _p(c, _f64p))
    return _by_rows(fn, a, N, threads)


def gemm_bf16_swiglu(a_bits, b_bits, threads=1):
    """h = silu(A . Bgate^T) * (A . Bup^T) in fp64; b_bits [2*Nh][K], gate rows first."""
    a, b = _c(a_bits, np.uint16), _c(b_bits, np.uint16)
    K = a.shape[1]
    Nh = b.shape[0] // 2

    def fn(ar, h):
        lib().orc_gemm_bf16_swiglu(_p(ar, _u16p), _p(b, _u16p), ar.shape[0], Nh, K, _p(h, _f64p))
    return _by_rows(fn, a, Nh, threads)


def bf16_rne_array(v):
    """fp64 array -> bf16 bit patterns (uint16), round to nearest even."""
    v = _c(v, np.float64)
    out = np.empty(v.shape, np.uint16)
    lib().orc_bf16_rne_n(_p(v, _f64p), v.size, _p(out, _u16p))
    return out


def block_forward(h_bits, k, w_down, w_router, w_shared13, w_out, w13, w13s, w2, w2s,
                  threads=0):
    """The composed latent-MoE block, step by step from the functions above
    ("Kimi K3.1 Pro at a glance": routed experts in a latent half the hidden
    width, two shared experts, BF16 router and latent projections; "Day 0
    Kimi-K3 ...", "Kimi-K3 Architecture and Weights": the hidden state is
    projected down to the latent before the experts). Every tensor that passes
    between steps is held in the format the library passes it in: x, the
    routed output and the shared experts' h as bf16, the logits as fp32.

      x      = bf16(h . w_down^T)                 [T][d]
      logits = fp32(h . w_router^T)               [T][E]
      y_lat  = moe_forward(x, logits)             [T][d] (bf16)
      hs     = bf16(silu(h . G^T) * (h . U^T))    [T][shared_I]
      out    = bf16([y_lat | hs] . w_out^T)       [T][hidden]

    h_bits bf16 patterns [T][hidden]; bf16 weights as bit patterns: w_down
    [d][hidden], w_router [E][hidden], w_shared13 [2 shared_I][hidden] (gate
    rows then up rows), w_out [hidden][d + shared_I]; routed weights as
    moe_forward. Returns dict(y (bf16 bits), y64 (fp64 before the last
    rounding), x, logits, ids, w, y_lat, hs)."""
    h = _c(h_bits, np.uint16)
    x = bf16_rne_array(gemm_bf16(h, w_down, threads))
    logits = gemm_bf16(h, w_router, threads).astype(np.float32)
    routed = moe_forward(x, logits, k, w13, w13s, w2, w2s, threads=threads)
    hs = bf16_rne_array(gemm_bf16_swiglu(h, w_shared13, threads))
    y64 = gemm_bf16(np.concatenate([routed["y"], hs], axis=1), w_out, threads)
    return dict(y=bf16_rne_array(y64), y64=y64, x=x, logits=logits, ids=routed["ids"],
                w=routed["w"], y_lat=routed["y"], hs=hs)


def expert_bytes(d, I):
    return lib().orc_expert_bytes(d, I)
