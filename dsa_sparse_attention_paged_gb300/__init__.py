"""Python binding of the GB300 DSA indexer decode library (``include/dsa.h``).

Argument marshalling only: every function here checks tensor dtypes, devices
and shapes, turns tensors into device pointers and calls the C ABI of
``_build/libdsa_gb300.so`` with the current CUDA stream.  All computation runs
in the library's sm_103a kernels; there is no Python or CPU fallback, and
importing this module fails loudly when the library has not been built.

Functions have the C names without the ``dsa_`` prefix.  Row r = b*next_n + j
of request b sees n_r = context_lens[b] - (next_n - 1 - j) keys.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libdsa_gb300.so")

NUM_BINS = 1024
MAX_TOPK = 2048
CAND_CAP = 8192
OUT_F32 = 0
OUT_F16 = 1
OUT_BF16 = 2
DEV_TIMEOUT = 0x1
DEV_BOUNDS = 0x2
INT32_MAX = 2**31 - 1
NOALLOC_MAX_ROWS = 64

_STATUS = {0: "DSA_OK", 1: "DSA_ERR_INVALID_ARG", 2: "DSA_ERR_UNSUPPORTED",
           3: "DSA_ERR_MISALIGNED", 4: "DSA_ERR_CUDA", 5: "DSA_ERR_WORKSPACE"}


class TopkProblem(ctypes.Structure):
    """``dsa_topk_problem``: one problem of ``coarse_hist_topk_batch``."""
    _fields_ = [("logits", ctypes.c_void_p), ("stride", ctypes.c_int64),
                ("context_lens", ctypes.c_void_p), ("histogram", ctypes.c_void_p),
                ("out_idx", ctypes.c_void_p), ("fallback_flags", ctypes.c_void_p),
                ("block_out_idx", ctypes.c_void_p), ("block_fallback_flags", ctypes.c_void_p),
                ("next_n", ctypes.c_int32), ("len_div", ctypes.c_int32), ("R", ctypes.c_int32),
                ("reset_histogram", ctypes.c_int32), ("k", ctypes.c_int32),
                ("block_k", ctypes.c_int32), ("block_page_table", ctypes.c_void_p),
                ("block_page_table_stride", ctypes.c_int64), ("block_page_size", ctypes.c_int32),
                ("block_phys", ctypes.c_void_p), ("block_valid_lens", ctypes.c_void_p)]


TOPK_BATCH_MAX = 4


class DecodeStepArgs(ctypes.Structure):
    """``dsa_decode_step_args``: the buffers and sizes of one decode step."""
    _fields_ = [("q", ctypes.c_void_p), ("kv_pages", ctypes.c_void_p),
                ("kscale", ctypes.c_void_p), ("weights", ctypes.c_void_p),
                ("page_table", ctypes.c_void_p), ("page_table_stride", ctypes.c_int64),
                ("context_lens", ctypes.c_void_p), ("B", ctypes.c_int32),
                ("next_n", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("k", ctypes.c_int32), ("kb", ctypes.c_int32),
                ("logits", ctypes.c_void_p), ("logits_stride", ctypes.c_int64),
                ("histogram", ctypes.c_void_p), ("topk_idx", ctypes.c_void_p),
                ("block_ids", ctypes.c_void_p), ("phys_blocks", ctypes.c_void_p),
                ("valid_lens", ctypes.c_void_p), ("sparse_scores", ctypes.c_void_p),
                ("sparse_idx", ctypes.c_void_p)]


class DSAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        cuda = lib.dsa_last_cuda_error() if lib is not None else 0
        super().__init__(f"{what}: {_STATUS.get(status, status)}"
                         + (f" (cuda error {cuda})" if status == 4 else ""))


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"CUDA library not built: {LIB_PATH} is missing. Build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` or "
            "`python dsa_sparse_attention_paged_gb300/build.py`.")
    L = ctypes.CDLL(LIB_PATH)
    P, i32, i64, sz, u32, u64 = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                 ctypes.c_size_t, ctypes.c_uint32, ctypes.c_uint64)
    sig = {
        "dsa_status_string": (ctypes.c_char_p, [i32]),
        "dsa_last_cuda_error": (i32, []),
        "dsa_version": (i32, []),
        "dsa_workspace_size": (sz, [i32]),
        "dsa_workspace_init": (i32, [P, sz, P]),
        "dsa_read_device_status": (i32, [P, P, ctypes.POINTER(u32)]),
        "dsa_paged_mqa_logits": (i32, [P, P, P, P, P, i64, P, i32, i32, i32, i32, i32, i32, P,
                                       i64, P, P, i64, i32, P, sz, P]),
        "dsa_paged_mqa_logits_mx": (i32, [P, P, P, P, P, i64, P, i32, i32, i32, i32, i32, i32,
                                          P, i64, P, P, sz, P]),
        "dsa_coarse_hist_topk": (i32, [P, i64, P, i32, i32, i32, P, i32, i32, P, P, P, sz, P]),
        "dsa_coarse_hist_topk_launches": (i32, [i64, i32]),
        "dsa_coarse_hist_topk_batch": (i32, [ctypes.POINTER(TopkProblem), i32, P, sz, P]),
        "dsa_coarse_hist_topk_batch_launches": (i32, [ctypes.POINTER(TopkProblem), i32]),
        "dsa_block_amax8": (i32, [P, i64, P, i32, i32, i32, P, i64, P, sz, P]),
        "dsa_sort_candidate_blocks": (i32, [P, i32, P, i32, i32, P, i64, i32, P, P, P, sz, P]),
        "dsa_sparse_mqa_logits": (i32, [P, P, P, P, P, i64, P, i32, i32, i32, i32, i32, i32, P,
                                        i32, P, P, P, i32, i64, P, sz, P]),
        "dsa_pair_units": (i32, [i32, i32]),
        "dsa_sort_candidate_blocks_paired": (i32, [P, i32, P, i32, i32, P, i64, i32, P, P, P, P,
                                                   P, P, sz, P]),
        "dsa_sparse_mqa_logits_paired": (i32, [P, P, P, P, P, i64, P, i32, i32, i32, i32, i32,
                                               i32, i32, P, P, P, P, P, i32, i64, P, sz, P]),
        "dsa_topk_fp16": (i32, [P, i64, P, i32, i32, P, i32, P, P, sz, P]),
        "dsa_topk_bf16": (i32, [P, i64, P, i32, i32, P, i32, P, P, sz, P]),
        "dsa_coarse_hist_topk_noalloc": (i32, [P, i64, P, i32, i32, i32, P, i32, i32, P, P, P]),
        "dsa_coarse_bins_range": (i32, [u32, i64, P, P]),
        "dsa_coarse_bin_key_ranges": (i32, [P, P]),
        "dsa_fp16_order_keys": (i32, [P, P, i64, P]),
        "dsa_bf16_order_keys": (i32, [P, P, i64, P]),
        "dsa_wait_timeout_selftest": (i32, [u64, P, sz, P]),
        "dsa_decode_step": (i32, [ctypes.POINTER(DecodeStepArgs), P, sz, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


lib = _load()


def _check(st: int, what: str):
    if st != 0:
        raise DSAError(st, what)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _req(t, dtype, name):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")


def _u8(t):
    return t.view(torch.uint8) if t.dtype == torch.float8_e4m3fn else t


class Workspace:
    """Caller-owned scratch buffer shared by all calls (zero-filled at creation;
    every completed call leaves it zeroed again)."""

    def __init__(self, max_rows: int, device=None):
        self.max_rows = int(max_rows)
        self.nbytes = int(lib.dsa_workspace_size(self.max_rows))
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8,
                               device=device if device is not None else "cuda")

    @property
    def ptr(self):
        return ctypes.c_void_p(self.buf.data_ptr())

    def init(self, stream=None):
        _check(lib.dsa_workspace_init(self.ptr, self.nbytes, _stream(stream)), "workspace_init")

    def status(self, stream=None) -> int:
        out = ctypes.c_uint32(0)
        _check(lib.dsa_read_device_status(self.ptr, _stream(stream), ctypes.byref(out)),
               "read_device_status")
        return int(out.value)


def workspace_size(max_rows: int) -> int:
    return int(lib.dsa_workspace_size(int(max_rows)))


def paged_mqa_logits(q, kv_pages, kscale, weights, page_table, context_lens, next_n, ws,
                     logits=None, logits_stride=None, histogram=None, amax=None,
                     amax_skip_if_blocks_le=0, stream=None):
    """Dense logits [B*next_n][stride] (dead columns untouched); when given,
    accumulate the coarse histogram and write the block maxima over 8 scores
    in the same pass.  Returns logits."""
    q, kv_pages = _u8(q), _u8(kv_pages)
    _req(q, torch.uint8, "q")
    _req(kv_pages, torch.uint8, "kv_pages")
    _req(kscale, torch.float32, "kscale")
    _req(weights, torch.float32, "weights")
    _req(page_table, torch.int32, "page_table")
    _req(context_lens, torch.int32, "context_lens")
    R, H, D = q.shape
    P, ps, D2 = kv_pages.shape
    B = context_lens.shape[0]
    if R != B * next_n or D2 != D:
        raise ValueError("shape mismatch between q, kv_pages and context_lens")
    if logits is None:
        stride = int(logits_stride) if logits_stride is not None else None
        if stride is None:
            raise ValueError("give logits or logits_stride")
        logits = torch.empty((R, stride), dtype=torch.float32, device=q.device)
    _req(logits, torch.float32, "logits")
    if histogram is not None:
        _req(histogram, torch.int32, "histogram")
    if amax is not None:
        _req(amax, torch.float32, "amax")
    for t in (q, kv_pages, kscale, weights, page_table, context_lens):
        assert t.is_contiguous()
    _check(lib.dsa_paged_mqa_logits(
        _p(q), _p(kv_pages), _p(kscale), _p(weights), _p(page_table), page_table.stride(0),
        _p(context_lens), B, next_n, H, D, ps, P, _p(logits), logits.stride(0), _p(histogram),
        _p(amax), amax.stride(0) if amax is not None else 0, int(amax_skip_if_blocks_le),
        ws.ptr, ws.nbytes, _stream(stream)), "paged_mqa_logits")
    return logits


def decode_step_args(q, kv_pages, kscale, weights, page_table, context_lens, next_n, k, kb,
                     logits, histogram, topk_idx, block_ids, phys_blocks, valid_lens,
                     sparse_scores, sparse_idx) -> DecodeStepArgs:
    """Checked argument block of ``decode_step`` (build it once and reuse it
    while the tensors stay the same: it holds their addresses)."""
    q, kv_pages = _u8(q), _u8(kv_pages)
    for t, dt, nm in ((q, torch.uint8, "q"), (kv_pages, torch.uint8, "kv_pages"),
                      (kscale, torch.float32, "kscale"), (weights, torch.float32, "weights"),
                      (page_table, torch.int32, "page_table"),
                      (context_lens, torch.int32, "context_lens"),
                      (logits, torch.float32, "logits"), (histogram, torch.int32, "histogram"),
                      (topk_idx, torch.int32, "topk_idx"), (block_ids, torch.int32, "block_ids"),
                      (phys_blocks, torch.int32, "phys_blocks"),
                      (valid_lens, torch.int32, "valid_lens"),
                      (sparse_scores, torch.float16, "sparse_scores"),
                      (sparse_idx, torch.int32, "sparse_idx")):
        _req(t, dt, nm)
    for t in (q, kv_pages, kscale, weights, page_table, context_lens, histogram, topk_idx,
              block_ids, phys_blocks, valid_lens, sparse_scores, sparse_idx):
        assert t.is_contiguous()
    R, H, D = q.shape
    P, ps, D2 = kv_pages.shape
    B = context_lens.shape[0]
    if R != B * next_n or D2 != D or H != 32 or D != 128:
        raise ValueError("shape mismatch between q, kv_pages and context_lens")
    if (tuple(histogram.shape) != (R, NUM_BINS) or tuple(topk_idx.shape) != (R, k)
            or tuple(block_ids.shape) != (R, kb) or tuple(phys_blocks.shape) != (R, kb)
            or tuple(valid_lens.shape) != (R,) or tuple(sparse_scores.shape) != (R, kb * 8)
            or tuple(sparse_idx.shape) != (R, k) or logits.shape[0] != R):
        raise ValueError("output shapes do not match B * next_n rows, k and kb")
    return DecodeStepArgs(
        q.data_ptr(), kv_pages.data_ptr(), kscale.data_ptr(), weights.data_ptr(),
        page_table.data_ptr(), page_table.stride(0), context_lens.data_ptr(), B, next_n, ps, P,
        k, kb, logits.data_ptr(), logits.stride(0), histogram.data_ptr(), topk_idx.data_ptr(),
        block_ids.data_ptr(), phys_blocks.data_ptr(), valid_lens.data_ptr(),
        sparse_scores.data_ptr(), sparse_idx.data_ptr())


def decode_step(args: DecodeStepArgs, ws, stream=None):
    """The whole two-level decode step in one library call (``dsa_decode_step``:
    dense logits + histogram, select with the sorted block table, sparse FP16
    logits, FP16 top-k), on the argument block from ``decode_step_args``."""
    _check(lib.dsa_decode_step(ctypes.byref(args), ws.ptr, ws.nbytes, _stream(stream)),
           "decode_step")


def paged_mqa_logits_mx(q, k_codes, k_exp, weights, page_table, context_lens, next_n, ws,
                        logits=None, logits_stride=None, histogram=None, stream=None):
    """Dense logits over an MXFP4 index-K cache: k_codes [P][ps][64] uint8
    (two E2M1 codes per byte, even dimension in the low nibble), k_exp
    [P][ps][4] uint8 (UE8M0, one per 32 dimensions).  Same outputs as
    paged_mqa_logits (dead columns untouched, optional histogram)."""
    q, k_codes, k_exp = _u8(q), _u8(k_codes), _u8(k_exp)
    _req(q, torch.uint8, "q")
    _req(k_codes, torch.uint8, "k_codes")
    _req(k_exp, torch.uint8, "k_exp")
    _req(weights, torch.float32, "weights")
    _req(page_table, torch.int32, "page_table")
    _req(context_lens, torch.int32, "context_lens")
    R, H, D = q.shape
    P, ps, Dh = k_codes.shape
    B = context_lens.shape[0]
    if R != B * next_n or 2 * Dh != D or tuple(k_exp.shape) != (P, ps, D // 32):
        raise ValueError("shape mismatch between q, k_codes, k_exp and context_lens")
    if logits is None:
        if logits_stride is None:
            raise ValueError("give logits or logits_stride")
        logits = torch.empty((R, int(logits_stride)), dtype=torch.float32, device=q.device)
    _req(logits, torch.float32, "logits")
    if histogram is not None:
        _req(histogram, torch.int32, "histogram")
    for t in (q, k_codes, k_exp, weights, page_table, context_lens):
        assert t.is_contiguous()
    _check(lib.dsa_paged_mqa_logits_mx(
        _p(q), _p(k_codes), _p(k_exp), _p(weights), _p(page_table), page_table.stride(0),
        _p(context_lens), B, next_n, H, D, ps, P, _p(logits), logits.stride(0), _p(histogram),
        ws.ptr, ws.nbytes, _stream(stream)), "paged_mqa_logits_mx")
    return logits


def coarse_hist_topk(logits, context_lens, next_n, k, ws, histogram=None, reset_histogram=False,
                     len_div=1, out=None, fallback_flags=None, R=None, stream=None):
    """Exact top-k columns per row ([R][k] int32, -1 padded, order unspecified)."""
    _req(logits, torch.float32, "logits")
    _req(context_lens, torch.int32, "context_lens")
    R = logits.shape[0] if R is None else R
    if out is None:
        out = torch.empty((R, k), dtype=torch.int32, device=logits.device)
    _req(out, torch.int32, "out")
    if histogram is not None:
        _req(histogram, torch.int32, "histogram")
    if fallback_flags is not None:
        _req(fallback_flags, torch.int32, "fallback_flags")
    _check(lib.dsa_coarse_hist_topk(
        _p(logits), logits.stride(0), _p(context_lens), next_n, len_div, R, _p(histogram),
        1 if reset_histogram else 0, k, _p(out), _p(fallback_flags), ws.ptr, ws.nbytes,
        _stream(stream)), "coarse_hist_topk")
    return out


def _topk_problem(logits, context_lens, next_n, k, histogram=None, reset_histogram=False,
                  len_div=1, out=None, fallback_flags=None, R=None, block_k=0, block_out=None,
                  block_fallback_flags=None, block_page_table=None, block_page_size=0,
                  block_phys=None, block_valid_lens=None):
    _req(logits, torch.float32, "logits")
    _req(context_lens, torch.int32, "context_lens")
    R = logits.shape[0] if R is None else R
    if out is None:
        out = torch.empty((R, k), dtype=torch.int32, device=logits.device)
    _req(out, torch.int32, "out")
    if histogram is not None:
        _req(histogram, torch.int32, "histogram")
    if fallback_flags is not None:
        _req(fallback_flags, torch.int32, "fallback_flags")
    if block_k and block_out is None:
        block_out = torch.empty((R, block_k), dtype=torch.int32, device=logits.device)
    if block_out is not None:
        _req(block_out, torch.int32, "block_out")
    if block_fallback_flags is not None:
        _req(block_fallback_flags, torch.int32, "block_fallback_flags")
    prob = TopkProblem(logits.data_ptr(), logits.stride(0), context_lens.data_ptr(),
                       histogram.data_ptr() if histogram is not None else None, out.data_ptr(),
                       fallback_flags.data_ptr() if fallback_flags is not None else None,
                       block_out.data_ptr() if block_out is not None else None,
                       block_fallback_flags.data_ptr() if block_fallback_flags is not None
                       else None,
                       int(next_n), int(len_div), int(R), 1 if reset_histogram else 0, int(k),
                       int(block_k))
    if block_page_table is not None:
        _req(block_page_table, torch.int32, "block_page_table")
        prob.block_page_table = block_page_table.data_ptr()
        prob.block_page_table_stride = block_page_table.stride(0)
        prob.block_page_size = int(block_page_size)
        if block_phys is not None:
            _req(block_phys, torch.int32, "block_phys")
            prob.block_phys = block_phys.data_ptr()
        if block_valid_lens is not None:
            _req(block_valid_lens, torch.int32, "block_valid_lens")
            prob.block_valid_lens = block_valid_lens.data_ptr()
    return prob, ((out, block_out) if block_k else out)


def coarse_hist_topk_batch(problems, ws, stream=None):
    """Several independent ``coarse_hist_topk`` problems (dicts of its keyword
    arguments, plus ``block_k`` / ``block_out`` / ``block_fallback_flags`` for
    the fused top block maxima, and ``block_page_table`` / ``block_page_size``
    / ``block_phys`` / ``block_valid_lens`` to have the block output written
    as the sorted block table) with one workspace sized for the sum of their
    rows; one launch when every row stride is at most 131072.  Returns per
    problem its output tensor, or (output, block output) with block_k."""
    if len(problems) > TOPK_BATCH_MAX:
        raise ValueError(f"coarse_hist_topk_batch: at most {TOPK_BATCH_MAX} problems")
    built = [_topk_problem(**p) for p in problems]
    arr = (TopkProblem * max(1, len(built)))(*[b[0] for b in built])
    _check(lib.dsa_coarse_hist_topk_batch(arr, len(built), ws.ptr, ws.nbytes, _stream(stream)),
           "coarse_hist_topk_batch")
    return [b[1] for b in built]


def coarse_hist_topk_batch_launches(strides_and_hist):
    """Kernel launches of ``coarse_hist_topk_batch`` for problems given as
    (row stride, has_histogram, rows) triples."""
    arr = (TopkProblem * max(1, len(strides_and_hist)))(
        *[TopkProblem(None, int(s), None, 1 if h else None, None, None, None, None, 1, 1, int(r),
                      0, 1, 0) for s, h, r in strides_and_hist])
    n = lib.dsa_coarse_hist_topk_batch_launches(arr, len(strides_and_hist))
    if n < 0:
        raise ValueError("coarse_hist_topk_batch_launches: invalid problems")
    return n


def block_amax8(logits, context_lens, next_n, ws, skip_if_blocks_le=0, amax=None,
                amax_stride=None, stream=None):
    _req(logits, torch.float32, "logits")
    _req(context_lens, torch.int32, "context_lens")
    R = logits.shape[0]
    if amax is None:
        amax_stride = (logits.stride(0) + 7) // 8 if amax_stride is None else amax_stride
        amax = torch.empty((R, amax_stride), dtype=torch.float32, device=logits.device)
    _req(amax, torch.float32, "amax")
    _check(lib.dsa_block_amax8(_p(logits), logits.stride(0), _p(context_lens), next_n, R,
                               skip_if_blocks_le, _p(amax), amax.stride(0), ws.ptr, ws.nbytes,
                               _stream(stream)), "block_amax8")
    return amax


def sort_candidate_blocks(block_ids, context_lens, next_n, page_table, page_size, ws,
                          phys_blocks=None, valid_lens=None, stream=None):
    """In place: block_ids [R][kb] -> ascending INT32_MAX-padded table."""
    _req(block_ids, torch.int32, "block_ids")
    R, kb = block_ids.shape
    _check(lib.dsa_sort_candidate_blocks(
        _p(block_ids), kb, _p(context_lens), next_n, R, _p(page_table), page_table.stride(0),
        page_size, _p(phys_blocks), _p(valid_lens), ws.ptr, ws.nbytes, _stream(stream)),
        "sort_candidate_blocks")
    return block_ids


def sparse_mqa_logits(q, kv_pages, kscale, weights, page_table, context_lens, next_n,
                      block_table, ws, out=None, out_dtype=OUT_F32, phys_blocks=None,
                      valid_lens=None, stream=None):
    """Sparse logits over the block table; with ``phys_blocks`` and
    ``valid_lens`` from ``sort_candidate_blocks`` the page-table reads are
    skipped (same results)."""
    q, kv_pages = _u8(q), _u8(kv_pages)
    R, H, D = q.shape
    P, ps, _ = kv_pages.shape
    B = context_lens.shape[0]
    kb = block_table.shape[1]
    if out is None:
        dt = {OUT_F32: torch.float32, OUT_F16: torch.float16, OUT_BF16: torch.bfloat16}[out_dtype]
        out = torch.empty((R, kb * 8), dtype=dt, device=q.device)
    _req(block_table, torch.int32, "block_table")
    for t, nm in ((phys_blocks, "phys_blocks"), (valid_lens, "valid_lens")):
        if t is not None:
            _req(t, torch.int32, nm)
    _check(lib.dsa_sparse_mqa_logits(
        _p(q), _p(kv_pages), _p(kscale), _p(weights), _p(page_table), page_table.stride(0),
        _p(context_lens), B, next_n, H, D, ps, P, _p(block_table), kb, _p(phys_blocks),
        _p(valid_lens), _p(out), out_dtype, out.stride(0), ws.ptr, ws.nbytes, _stream(stream)),
        "sparse_mqa_logits")
    return out


def pair_units(B: int, next_n: int) -> int:
    """Units of the paired sparse pass: B * ceil(next_n / 2)."""
    return int(lib.dsa_pair_units(B, next_n))


def sort_candidate_blocks_paired(block_ids, context_lens, next_n, page_table, page_size, ws,
                                 valid_lens, union, phys_blocks=None, stream=None):
    """``sort_candidate_blocks`` for every row (in place, same tables) plus the
    union of each unit's two tables.  ``union`` is (union_phys [U][2kb],
    union_pos [U][2kb], union_len [U]) int32, filled; returns it."""
    _req(block_ids, torch.int32, "block_ids")
    R, kb = block_ids.shape
    B = context_lens.shape[0]
    uphys, upos, ulen = union
    U = pair_units(B, next_n)
    for t, nm, shp in ((uphys, "union_phys", (U, 2 * kb)), (upos, "union_pos", (U, 2 * kb)),
                       (ulen, "union_len", (U,)), (valid_lens, "valid_lens", (R,))):
        _req(t, torch.int32, nm)
        if tuple(t.shape) != shp or not t.is_contiguous():
            raise ValueError(f"{nm}: expected a contiguous {shp} tensor")
    if phys_blocks is not None:
        _req(phys_blocks, torch.int32, "phys_blocks")
    _check(lib.dsa_sort_candidate_blocks_paired(
        _p(block_ids), kb, _p(context_lens), next_n, B, _p(page_table), page_table.stride(0),
        page_size, _p(phys_blocks), _p(valid_lens), _p(uphys), _p(upos), _p(ulen), ws.ptr,
        ws.nbytes, _stream(stream)), "sort_candidate_blocks_paired")
    return union


def sparse_mqa_logits_paired(q, kv_pages, kscale, weights, page_table, context_lens, next_n,
                             kb, union, valid_lens, ws, out=None, out_dtype=OUT_F32,
                             stream=None):
    """Sparse logits of every row, two rows of a request per K pass (bitwise
    the output of ``sparse_mqa_logits`` with physical blocks)."""
    q, kv_pages = _u8(q), _u8(kv_pages)
    R, H, D = q.shape
    P, ps, _ = kv_pages.shape
    B = context_lens.shape[0]
    uphys, upos, ulen = union
    if out is None:
        dt = {OUT_F32: torch.float32, OUT_F16: torch.float16, OUT_BF16: torch.bfloat16}[out_dtype]
        out = torch.empty((R, kb * 8), dtype=dt, device=q.device)
    U = pair_units(B, next_n)
    for t, nm, shp in ((uphys, "union_phys", (U, 2 * kb)), (upos, "union_pos", (U, 2 * kb)),
                       (ulen, "union_len", (U,)), (valid_lens, "valid_lens", (R,))):
        _req(t, torch.int32, nm)
        if tuple(t.shape) != shp or not t.is_contiguous():
            raise ValueError(f"{nm}: expected a contiguous {shp} tensor")
    _check(lib.dsa_sparse_mqa_logits_paired(
        _p(q), _p(kv_pages), _p(kscale), _p(weights), _p(page_table), page_table.stride(0),
        _p(context_lens), B, next_n, H, D, ps, P, kb, _p(uphys), _p(upos), _p(ulen),
        _p(valid_lens), _p(out), out_dtype, out.stride(0), ws.ptr, ws.nbytes, _stream(stream)),
        "sparse_mqa_logits_paired")
    return out


def topk_fp16(scores, valid_lens, k, ws, block_table=None, out=None, stream=None):
    """Top-k over FP16 scores (torch.float16 or raw uint16 bits)."""
    s = scores.view(torch.uint16) if scores.dtype == torch.float16 else scores
    _req(s, torch.uint16, "scores")
    R = s.shape[0]
    if out is None:
        out = torch.empty((R, k), dtype=torch.int32, device=s.device)
    kb = 0 if block_table is None else block_table.shape[1]
    _check(lib.dsa_topk_fp16(_p(s), s.stride(0), _p(valid_lens), R, k, _p(block_table), kb,
                             _p(out), ws.ptr, ws.nbytes, _stream(stream)), "topk_fp16")
    return out


def topk_bf16(scores, valid_lens, k, ws, block_table=None, out=None, stream=None):
    """Top-k over BF16 scores (torch.bfloat16 or raw uint16 bits)."""
    s = scores.view(torch.uint16) if scores.dtype == torch.bfloat16 else scores
    _req(s, torch.uint16, "scores")
    R = s.shape[0]
    if out is None:
        out = torch.empty((R, k), dtype=torch.int32, device=s.device)
    kb = 0 if block_table is None else block_table.shape[1]
    _check(lib.dsa_topk_bf16(_p(s), s.stride(0), _p(valid_lens), R, k, _p(block_table), kb,
                             _p(out), ws.ptr, ws.nbytes, _stream(stream)), "topk_bf16")
    return out


def coarse_bin_key_ranges(stream=None):
    """[1025][2] uint32 (as int64): lowest and highest order key of each coarse
    bin as the select computes them (bin 1024: an empty range)."""
    out = torch.zeros(2 * 1025, dtype=torch.int32, device="cuda")
    _check(lib.dsa_coarse_bin_key_ranges(_p(out), _stream(stream)), "coarse_bin_key_ranges")
    return (out.cpu().to(torch.int64) & 0xFFFFFFFF).view(1025, 2)


def coarse_bins_range(start: int, count: int, out=None, stream=None):
    if out is None:
        out = torch.empty(count, dtype=torch.int16, device="cuda")
    _check(lib.dsa_coarse_bins_range(ctypes.c_uint32(start), count, _p(out), _stream(stream)),
           "coarse_bins_range")
    return out


def fp16_order_keys(x, out=None, stream=None):
    s = x.view(torch.uint16) if x.dtype == torch.float16 else x
    if out is None:
        out = torch.empty_like(s)
    _check(lib.dsa_fp16_order_keys(_p(s), _p(out), s.numel(), _stream(stream)),
           "fp16_order_keys")
    return out


def bf16_order_keys(x, out=None, stream=None):
    s = x.view(torch.uint16) if x.dtype == torch.bfloat16 else x
    if out is None:
        out = torch.empty_like(s)
    _check(lib.dsa_bf16_order_keys(_p(s), _p(out), s.numel(), _stream(stream)),
           "bf16_order_keys")
    return out


def wait_timeout_selftest(limit_cycles: int, ws, stream=None):
    _check(lib.dsa_wait_timeout_selftest(ctypes.c_uint64(limit_cycles), ws.ptr, ws.nbytes,
                                         _stream(stream)), "wait_timeout_selftest")


def coarse_hist_topk_launches(stride, has_histogram):
    """Kernel launches one coarse_hist_topk call makes on rows of ``stride``."""
    n = lib.dsa_coarse_hist_topk_launches(int(stride), 1 if has_histogram else 0)
    if n < 0:
        raise ValueError(f"coarse_hist_topk_launches: invalid stride {stride}")
    return n


def coarse_hist_topk_noalloc(logits, context_lens, next_n, k, histogram=None,
                             reset_histogram=False, len_div=1, out=None, fallback_flags=None,
                             R=None, stream=None):
    """coarse_hist_topk for callers that cannot allocate device memory: the
    scratch lives in a fixed array inside the library (at most NOALLOC_MAX_ROWS
    rows; calls that overlap on the GPU race on it).  ``out`` and
    ``fallback_flags`` are the caller's own buffers."""
    _req(logits, torch.float32, "logits")
    _req(context_lens, torch.int32, "context_lens")
    R = logits.shape[0] if R is None else R
    if out is None:
        out = torch.empty((R, k), dtype=torch.int32, device=logits.device)
    _req(out, torch.int32, "out")
    _check(lib.dsa_coarse_hist_topk_noalloc(
        _p(logits), logits.stride(0), _p(context_lens), next_n, len_div, R, _p(histogram),
        1 if reset_histogram else 0, k, _p(out), _p(fallback_flags), _stream(stream)),
        "coarse_hist_topk_noalloc")
    return out
