"""Python marshalling for the C oracle in ``dsa_oracle.c``.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the bench's CPU
baseline leg may import this module; the library's product path never does.
The oracle shares no code with the CUDA library.  This wrapper only converts
numpy arrays to pointers; every step of the arithmetic is in the C file, which
cites the pages section by section.

The shared object is compiled on first use (``gcc -O2 -ffp-contract=off``:
no fused multiply-adds, so x86-64 and aarch64 hosts round identically).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD_DIR, "liboracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (atomic replace)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_BUILD_DIR)
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    i64 = ctypes.c_int64
    i32 = ctypes.c_int
    lib.o_e4m3_to_double.restype = ctypes.c_double
    lib.o_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.o_e4m3_table.argtypes = [P]
    lib.o_fp16_rn_bits.restype = ctypes.c_uint16
    lib.o_fp16_rn_bits.argtypes = [ctypes.c_float]
    lib.o_fp16_bits_to_double.restype = ctypes.c_double
    lib.o_fp16_bits_to_double.argtypes = [ctypes.c_uint16]
    lib.o_coarse_bin.restype = ctypes.c_int32
    lib.o_coarse_bin.argtypes = [ctypes.c_float]
    lib.o_paged_mqa_logits.argtypes = [P, P, P, P, P, i64, P, i32, i32, i32, i32, i32, P, i64]
    lib.o_logits_at.argtypes = [P, P, P, P, P, i64, i32, i32, i32, i32, P, P, i64, P]
    lib.o_histogram_accumulate.argtypes = [P, i64, P, i32, P]
    lib.o_topk_row.restype = i64
    lib.o_topk_row.argtypes = [P, i64, i64, P]
    lib.o_topk.argtypes = [P, i64, P, i32, i64, P]
    lib.o_block_amax8.argtypes = [P, i64, P, i32, i64, P, i64]
    lib.o_block_table.argtypes = [P, i64, P, P, i32, i32, P, i64, i32, P, P, P]
    lib.o_sparse_logits.argtypes = [P, P, P, P, P, i64, P, P, i32, i32, i32, i32, P, i32, P, i64]
    lib.o_topk_fp16.argtypes = [P, i64, P, i32, i64, P, i32, P]
    lib.o_fp16_rn_sweep.argtypes = [ctypes.c_uint64, ctypes.c_uint64, P]
    lib.o_coarse_bin_sweep.argtypes = [ctypes.c_uint64, ctypes.c_uint64, P]
    lib.o_coarse_bins.argtypes = [P, i64, P]
    lib.o_fp16_rn_array.argtypes = [P, i64, P]
    lib.o_bf16_rn_bits.restype = ctypes.c_uint16
    lib.o_bf16_rn_bits.argtypes = [ctypes.c_float]
    lib.o_bf16_bits_to_double.restype = ctypes.c_double
    lib.o_bf16_bits_to_double.argtypes = [ctypes.c_uint16]
    lib.o_bf16_rn_array.argtypes = [P, i64, P]
    lib.o_bf16_rn_sweep.argtypes = [ctypes.c_uint64, ctypes.c_uint64, P]
    lib.o_topk_bf16.argtypes = [P, i64, P, i32, i64, P, i32, P]
    lib.o_pair_union.argtypes = [P, P, i32, i32, i32, P, P, P]
    lib.o_e2m1.restype = ctypes.c_double
    lib.o_e2m1.argtypes = [ctypes.c_uint8]
    lib.o_ue8m0.restype = ctypes.c_double
    lib.o_ue8m0.argtypes = [ctypes.c_uint8]
    lib.o_paged_mqa_logits_mx.argtypes = [P, P, P, P, P, i64, P, i32, i32, i32, i32, i32, P,
                                          i64]
    lib.o_logits_at_mx.argtypes = [P, P, P, P, P, i64, i32, i32, i32, i32, P, P, i64, P]
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# scalar helpers

def e4m3_table() -> np.ndarray:
    out = np.zeros(256, dtype=np.float64)
    _load().o_e4m3_table(_ptr(out))
    return out


def fp16_rn_bits(x: float) -> int:
    return int(_load().o_fp16_rn_bits(ctypes.c_float(x)))


def fp16_bits_to_double(h: int) -> float:
    return float(_load().o_fp16_bits_to_double(ctypes.c_uint16(h)))


def bf16_rn_bits(x: float) -> int:
    return int(_load().o_bf16_rn_bits(ctypes.c_float(x)))


def bf16_bits_to_double(h: int) -> float:
    return float(_load().o_bf16_bits_to_double(ctypes.c_uint16(h)))


def bf16_rn_sweep(start: int, count: int) -> np.ndarray:
    out = np.empty(count, dtype=np.uint16)
    _load().o_bf16_rn_sweep(ctypes.c_uint64(start), ctypes.c_uint64(count), _ptr(out))
    return out


def bf16_rn_array(x: np.ndarray) -> np.ndarray:
    """bfloat16 round-to-nearest-even bit patterns of a float32 array."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().o_bf16_rn_array(_ptr(x), x.size, _ptr(out))
    return out


def coarse_bin(x: float) -> int:
    return int(_load().o_coarse_bin(ctypes.c_float(x)))


def fp16_rn_sweep(start: int, count: int) -> np.ndarray:
    out = np.empty(count, dtype=np.uint16)
    _load().o_fp16_rn_sweep(ctypes.c_uint64(start), ctypes.c_uint64(count), _ptr(out))
    return out


def coarse_bin_sweep(start: int, count: int) -> np.ndarray:
    out = np.empty(count, dtype=np.int16)
    _load().o_coarse_bin_sweep(ctypes.c_uint64(start), ctypes.c_uint64(count), _ptr(out))
    return out


def coarse_bins(x: np.ndarray) -> np.ndarray:
    """Bin every element of a float32 array; -1 marks NaN."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, dtype=np.int16)
    _load().o_coarse_bins(_ptr(x), x.size, _ptr(out))
    return out


def fp16_rn_array(x: np.ndarray) -> np.ndarray:
    """IEEE binary16 round-to-nearest-even bit patterns of a float32 array."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().o_fp16_rn_array(_ptr(x), x.size, _ptr(out))
    return out


# --------------------------------------------------------------------------
# the path's operations

def row_lens(context_lens: np.ndarray, next_n: int) -> np.ndarray:
    """n_r = C_b - (next_n - 1 - j) for row r = b*next_n + j (reading R1)."""
    c = np.asarray(context_lens, dtype=np.int64)
    j = np.arange(next_n, dtype=np.int64)
    return (c[:, None] - (next_n - 1 - j)[None, :]).reshape(-1)


def paged_mqa_logits(q, kv, kscale, weights, page_table, context_lens, next_n,
                     page_size, logits_stride=None, fill=np.nan) -> np.ndarray:
    """Dense logits [R][stride] float32; dead columns keep ``fill``."""
    q = _c(q, np.uint8)
    kv = _c(kv, np.uint8)
    kscale = _c(kscale, np.float32)
    weights = _c(weights, np.float32)
    page_table = _c(page_table, np.int32)
    context_lens = _c(context_lens, np.int32)
    B = context_lens.shape[0]
    R, H, D = q.shape
    assert R == B * next_n
    if logits_stride is None:
        logits_stride = int(context_lens.max()) if B else 0
    out = np.full((R, max(logits_stride, 1)), fill, dtype=np.float32)
    _load().o_paged_mqa_logits(_ptr(q), _ptr(kv), _ptr(kscale), _ptr(weights),
                               _ptr(page_table), page_table.shape[1], _ptr(context_lens),
                               B, next_n, H, D, page_size, _ptr(out), out.shape[1])
    return out


def e2m1(code: int) -> float:
    """Value of a 4-bit E2M1 code (MXFP4 element)."""
    return _load().o_e2m1(code)


def ue8m0(e: int) -> float:
    """Value of an 8-bit UE8M0 block exponent."""
    return _load().o_ue8m0(e)


def paged_mqa_logits_mx(q, k_codes, k_exp, weights, page_table, context_lens, next_n,
                        page_size, logits_stride=None, fill=np.nan) -> np.ndarray:
    """Dense logits over an MXFP4 paged key cache: k_codes [P][page][D/2]
    (two E2M1 codes per byte, even dimension low), k_exp [P][page][D/32]
    (UE8M0); [R][stride] float32, dead columns keep ``fill``."""
    q = _c(q, np.uint8)
    k_codes = _c(k_codes, np.uint8)
    k_exp = _c(k_exp, np.uint8)
    weights = _c(weights, np.float32)
    page_table = _c(page_table, np.int32)
    context_lens = _c(context_lens, np.int32)
    B = context_lens.shape[0]
    R, H, D = q.shape
    assert R == B * next_n and k_codes.shape[-1] * 2 == D and k_exp.shape[-1] * 32 == D
    if logits_stride is None:
        logits_stride = int(context_lens.max()) if B else 0
    out = np.full((R, max(logits_stride, 1)), fill, dtype=np.float32)
    _load().o_paged_mqa_logits_mx(_ptr(q), _ptr(k_codes), _ptr(k_exp), _ptr(weights),
                                  _ptr(page_table), page_table.shape[1], _ptr(context_lens), B,
                                  next_n, H, D, page_size, _ptr(out), out.shape[1])
    return out


def logits_at_mx(q, k_codes, k_exp, weights, page_table, next_n, page_size, rows,
                 cols) -> np.ndarray:
    """MXFP4-key logits at (rows[i], cols[i]) pairs, one by one."""
    q = _c(q, np.uint8)
    k_codes = _c(k_codes, np.uint8)
    k_exp = _c(k_exp, np.uint8)
    weights = _c(weights, np.float32)
    page_table = _c(page_table, np.int32)
    rows = _c(rows, np.int64)
    cols = _c(cols, np.int64)
    R, H, D = q.shape
    out = np.empty(rows.shape[0], np.float32)
    _load().o_logits_at_mx(_ptr(q), _ptr(k_codes), _ptr(k_exp), _ptr(weights),
                           _ptr(page_table), page_table.shape[1], next_n, H, D, page_size,
                           _ptr(rows), _ptr(cols), rows.shape[0], _ptr(out))
    return out


def logits_at(q, kv, kscale, weights, page_table, next_n, page_size, rows, cols) -> np.ndarray:
    q = _c(q, np.uint8)
    kv = _c(kv, np.uint8)
    kscale = _c(kscale, np.float32)
    weights = _c(weights, np.float32)
    page_table = _c(page_table, np.int32)
    rows = _c(rows, np.int64)
    cols = _c(cols, np.int64)
    R, H, D = q.shape
    out = np.empty(rows.size, dtype=np.float32)
    _load().o_logits_at(_ptr(q), _ptr(kv), _ptr(kscale), _ptr(weights), _ptr(page_table),
                        page_table.shape[1], next_n, H, D, page_size, _ptr(rows), _ptr(cols),
                        rows.size, _ptr(out))
    return out


def histogram(logits, row_lens_, hist_in=None) -> np.ndarray:
    logits = _c(logits, np.float32)
    rl = _c(row_lens_, np.int64)
    R = logits.shape[0]
    hist = np.zeros((R, 1024), np.int32) if hist_in is None else _c(hist_in, np.int32).copy()
    _load().o_histogram_accumulate(_ptr(logits), logits.shape[1], _ptr(rl), R, _ptr(hist))
    return hist


def topk(logits, row_lens_, k) -> np.ndarray:
    """[R][k] int32, (value desc, column asc) order, -1 padded."""
    logits = _c(logits, np.float32)
    rl = _c(row_lens_, np.int64)
    R = logits.shape[0]
    out = np.empty((R, k), np.int32)
    _load().o_topk(_ptr(logits), logits.shape[1], _ptr(rl), R, k, _ptr(out))
    return out


def block_amax8(logits, row_lens_, skip_le=0, amax_stride=None, fill=np.nan) -> np.ndarray:
    logits = _c(logits, np.float32)
    rl = _c(row_lens_, np.int64)
    R = logits.shape[0]
    if amax_stride is None:
        amax_stride = max(1, (int(rl.max()) + 7) // 8 if R else 1)
    out = np.full((R, amax_stride), fill, np.float32)
    _load().o_block_amax8(_ptr(logits), logits.shape[1], _ptr(rl), R, skip_le, _ptr(out),
                          amax_stride)
    return out


def block_table(amax, row_lens_, row_to_req, kb, page_table, page_size):
    """Returns (table [R][kb], phys [R][kb], valid_len [R])."""
    amax = _c(amax, np.float32)
    rl = _c(row_lens_, np.int64)
    rtr = _c(row_to_req, np.int32)
    page_table = _c(page_table, np.int32)
    R = rl.shape[0]
    table = np.empty((R, kb), np.int32)
    phys = np.empty((R, kb), np.int32)
    vl = np.empty(R, np.int32)
    _load().o_block_table(_ptr(amax), amax.shape[1], _ptr(rl), _ptr(rtr), R, kb,
                          _ptr(page_table), page_table.shape[1], page_size, _ptr(table),
                          _ptr(phys), _ptr(vl))
    return table, phys, vl


def sparse_logits(q, kv, kscale, weights, page_table, row_lens_, row_to_req, page_size,
                  table) -> np.ndarray:
    q = _c(q, np.uint8)
    kv = _c(kv, np.uint8)
    kscale = _c(kscale, np.float32)
    weights = _c(weights, np.float32)
    page_table = _c(page_table, np.int32)
    rl = _c(row_lens_, np.int64)
    rtr = _c(row_to_req, np.int32)
    table = _c(table, np.int32)
    R, H, D = q.shape
    kb = table.shape[1]
    out = np.empty((R, kb * 8), np.float32)
    _load().o_sparse_logits(_ptr(q), _ptr(kv), _ptr(kscale), _ptr(weights), _ptr(page_table),
                            page_table.shape[1], _ptr(rl), _ptr(rtr), R, H, D, page_size,
                            _ptr(table), kb, _ptr(out), out.shape[1])
    return out


def pair_union(table, phys, next_n):
    """Row pairing of the sparse pass: (union_phys [U][2kb], union_pos
    [U][2kb], union_len [U]) for U = requests * ceil(next_n / 2) units."""
    table = _c(table, np.int32)
    phys = _c(phys, np.int32)
    R, kb = table.shape
    U = (R // next_n) * ((next_n + 1) // 2)
    up = np.empty((U, 2 * kb), np.int32)
    uq = np.empty((U, 2 * kb), np.int32)
    ul = np.empty(U, np.int32)
    _load().o_pair_union(_ptr(table), _ptr(phys), R, next_n, kb, _ptr(up), _ptr(uq), _ptr(ul))
    return up, uq, ul


def topk_fp16(scores_u16, valid_len, k, table=None) -> np.ndarray:
    s = _c(scores_u16, np.uint16)
    vl = _c(valid_len, np.int32)
    R = s.shape[0]
    out = np.empty((R, k), np.int32)
    if table is not None:
        table = _c(table, np.int32)
        tp, kb = _ptr(table), table.shape[1]
    else:
        tp, kb = ctypes.c_void_p(0), 0
    _load().o_topk_fp16(_ptr(s), s.shape[1], _ptr(vl), R, k, tp, kb, _ptr(out))
    return out



def topk_bf16(scores_u16, valid_len, k, table=None) -> np.ndarray:
    s = _c(scores_u16, np.uint16)
    vl = _c(valid_len, np.int32)
    R = s.shape[0]
    out = np.empty((R, k), np.int32)
    if table is not None:
        table = _c(table, np.int32)
        tp, kb = _ptr(table), table.shape[1]
    else:
        tp, kb = ctypes.c_void_p(0), 0
    _load().o_topk_bf16(_ptr(s), s.shape[1], _ptr(vl), R, k, tp, kb, _ptr(out))
    return out
