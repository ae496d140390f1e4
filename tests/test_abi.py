"""CPU-side checks of the C ABI: the library loads and exports every function
include/dsa.h declares, and host-side argument checks reject bad calls with
the documented status before anything touches the GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HDR = os.path.join(ROOT, "include", "dsa.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    import dsa_sparse_attention_paged_gb300 as D
    return D.lib


def declared():
    src = open(HDR).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_sizes(lib):
    assert lib.dsa_status_string(0) == b"DSA_OK"
    assert lib.dsa_status_string(2) == b"DSA_ERR_UNSUPPORTED"
    assert lib.dsa_version() >= 10000
    s1, s32 = lib.dsa_workspace_size(1), lib.dsa_workspace_size(32)
    assert s32 > s1 > 0 and s32 % 256 == 0
    # per row: 16 B counters + 8192 x 8 B candidates + 4 KiB histogram + 16 KiB fine histogram
    assert s32 - s1 >= 31 * (16 + 8192 * 8 + 4096 + 16384) - 1024


A16 = ctypes.c_void_p(0x10000)     # aligned, never dereferenced: checks fail first
MIS = ctypes.c_void_p(0x10004)


def paged(lib, **kw):
    a = dict(q=A16, kv=A16, ks=A16, w=A16, pt=A16, pts=4, ctx=A16, B=2, nn=1, H=32, D=128,
             ps=64, P=10, out=A16, ostride=256, hist=None, amax=None, astride=0, askip=0,
             ws=ctypes.c_void_p(0x20000), wsb=4096, st=None)
    a.update(kw)
    return lib.dsa_paged_mqa_logits(a["q"], a["kv"], a["ks"], a["w"], a["pt"], a["pts"], a["ctx"],
                                    a["B"], a["nn"], a["H"], a["D"], a["ps"], a["P"], a["out"],
                                    a["ostride"], a["hist"], a["amax"], a["astride"], a["askip"],
                                    a["ws"], a["wsb"], a["st"])


def sparse(lib, **kw):
    a = dict(q=A16, kv=A16, ks=A16, w=A16, pt=A16, pts=4, ctx=A16, B=2, nn=1, H=32, D=128,
             ps=64, P=10, bt=A16, kb=64, phys=None, vl=None, out=A16, dt=0, ostride=512,
             ws=ctypes.c_void_p(0x20000), wsb=4096, st=None)
    a.update(kw)
    return lib.dsa_sparse_mqa_logits(a["q"], a["kv"], a["ks"], a["w"], a["pt"], a["pts"],
                                     a["ctx"], a["B"], a["nn"], a["H"], a["D"], a["ps"], a["P"],
                                     a["bt"], a["kb"], a["phys"], a["vl"], a["out"], a["dt"],
                                     a["ostride"], a["ws"], a["wsb"], a["st"])


def test_sparse_logits_argument_checks(lib):
    assert sparse(lib, phys=A16) == 1          # physical blocks without live lengths
    assert sparse(lib, vl=A16) == 1
    assert sparse(lib, kb=40) == 2
    assert sparse(lib, ostride=100) == 1
    assert sparse(lib, bt=None) == 1


def test_paged_logits_argument_checks(lib):
    assert paged(lib, nn=5) == 2
    assert paged(lib, nn=0) == 2
    assert paged(lib, H=64) == 2
    assert paged(lib, D=64) == 2
    assert paged(lib, ps=32) == 2
    assert paged(lib, q=MIS) == 3
    assert paged(lib, kv=MIS) == 3
    assert paged(lib, hist=ctypes.c_void_p(0x10004)) == 3
    assert paged(lib, ws=None) == 5
    assert paged(lib, wsb=16) == 5
    assert paged(lib, q=None) == 1
    assert paged(lib, B=-1) == 1
    assert paged(lib, ostride=0) == 1
    assert paged(lib, amax=A16, astride=0) == 1
    assert paged(lib, B=0) == 0          # nothing to do, nothing launched


def test_topk_and_block_argument_checks(lib):
    ws = ctypes.c_void_p(0x20000)
    big = lib.dsa_workspace_size(4)
    f = lib.dsa_coarse_hist_topk
    assert f(A16, 128, A16, 1, 1, 4, None, 0, 0, A16, None, ws, big, None) == 2      # k = 0
    assert f(A16, 128, A16, 1, 1, 4, None, 0, 4096, A16, None, ws, big, None) == 2   # k > 2048
    assert f(A16, 128, A16, 1, 1, 4, None, 0, 16, A16, None, ws, 1024, None) == 5    # too small
    assert f(A16, 128, A16, 1, 1, 0, None, 0, 16, A16, None, ws, big, None) == 0     # R = 0
    assert f(A16, 128, A16, 1, 0, 4, None, 0, 16, A16, None, ws, big, None) == 1     # len_div
    g = lib.dsa_block_amax8
    assert g(MIS, 128, A16, 1, 2, 0, A16, 16, ws, 4096, None) == 3
    assert g(A16, 130, A16, 1, 2, 0, A16, 16, ws, 4096, None) == 3
    h = lib.dsa_sort_candidate_blocks
    assert h(A16, 8192, A16, 1, 2, A16, 4, 64, None, None, ws, 4096, None) == 2
    assert h(A16, 512, A16, 1, 2, A16, 4, 12, None, None, ws, 4096, None) == 2
    s = lib.dsa_sparse_mqa_logits
    assert s(A16, A16, A16, A16, A16, 4, A16, 2, 1, 32, 128, 64, 10, A16, 500, None, None, A16,
             0, 4000, ws, 4096, None) == 2  # kb not a multiple of 16
    assert s(A16, A16, A16, A16, A16, 4, A16, 2, 1, 32, 128, 64, 10, A16, 512, None, None, A16,
             0, 100, ws, 4096, None) == 1  # out_stride < kb * 8
    t = lib.dsa_topk_fp16
    assert t(A16, 4097, A16, 2, 16, None, 0, A16, ws, 4096, None) == 3  # odd stride
    assert t(A16, 4096, A16, 2, 0, None, 0, A16, ws, 4096, None) == 2


def test_topk_launch_count_follows_the_dispatch():
    """Host-only query: one cluster launch up to 131072 scores per row, else
    the multi-CTA passes (plus the histogram build without a histogram)."""
    import dsa_sparse_attention_paged_gb300 as D
    assert D.coarse_hist_topk_launches(1, True) == 1
    assert D.coarse_hist_topk_launches(131072, True) == 1
    assert D.coarse_hist_topk_launches(131072, False) == 1
    assert D.coarse_hist_topk_launches(131073, True) == 2
    assert D.coarse_hist_topk_launches(1 << 20, False) == 3
    with pytest.raises(ValueError):
        D.coarse_hist_topk_launches(0, True)


def test_topk_problem_layout_and_batch_launch_count():
    """dsa_topk_problem is 88 bytes (eight 8-byte fields, six int32); the batch
    runs in one launch when every row stride is at most 131072."""
    import ctypes
    import dsa_sparse_attention_paged_gb300 as D
    assert ctypes.sizeof(D.TopkProblem) == 128
    assert D.TopkProblem.next_n.offset == 64 and D.TopkProblem.block_k.offset == 84
    assert D.TopkProblem.block_page_table.offset == 88
    assert D.TopkProblem.block_page_table_stride.offset == 96
    assert D.TopkProblem.block_page_size.offset == 104
    assert D.TopkProblem.block_phys.offset == 112 and D.TopkProblem.block_valid_lens.offset == 120
    n = D.coarse_hist_topk_batch_launches
    assert n([(131072, True, 32), (16384, False, 32)]) == 1
    assert n([(200000, True, 2), (16384, False, 2)]) == 2 + 1
    assert n([(200000, True, 0), (16384, False, 2)]) == 1  # empty problems are skipped
    assert n([(16384, False, 0)]) == 0
    with pytest.raises(ValueError):
        n([(100, True, 1)] * 5)


def test_batch_block_output_argument_checks(lib):
    """Block outputs need an output pointer, block_k <= 2048, rows of scores
    (len_div 1) and rows a cluster takes (stride <= 131072); all refused
    before anything is launched."""
    import ctypes
    import dsa_sparse_attention_paged_gb300 as D

    def prob(**kw):
        f = dict(logits=0x10000, stride=4096, context_lens=0x10000, histogram=None,
                 out_idx=0x10000, fallback_flags=None, block_out_idx=0x10000,
                 block_fallback_flags=None, next_n=1, len_div=1, R=2, reset_histogram=0,
                 k=64, block_k=16)
        f.update(kw)
        return D.TopkProblem(**f)

    def call(*ps):
        arr = (D.TopkProblem * len(ps))(*ps)
        return lib.dsa_coarse_hist_topk_batch(arr, len(ps), ctypes.c_void_p(0x20000), 1 << 30,
                                              None)
    assert call(prob(block_out_idx=None)) == 1
    assert call(prob(block_k=-1)) == 1
    assert call(prob(block_k=4096)) == 2
    assert call(prob(len_div=8)) == 2
    assert call(prob(stride=200000)) == 2
    assert call(prob(stride=1000), prob(stride=200000, block_k=0, block_out_idx=None)) == 2


def test_paired_sort_and_sparse_argument_checks(lib):
    """The paired calls need the union buffers and live lengths; kb as for
    the unpaired calls; all refused before anything is launched."""
    ws = ctypes.c_void_p(0x20000)
    assert lib.dsa_pair_units(5, 4) == 10 and lib.dsa_pair_units(5, 3) == 10
    assert lib.dsa_pair_units(2, 1) == 2 and lib.dsa_pair_units(-1, 2) == 0
    h = lib.dsa_sort_candidate_blocks_paired
    ok = dict(ids=A16, kb=64, ctx=A16, nn=2, B=2, pt=A16, pts=4, ps=64, phys=None, vl=A16,
              up=A16, uq=A16, ul=A16)

    def sort(**kw):
        a = dict(ok)
        a.update(kw)
        return h(a["ids"], a["kb"], a["ctx"], a["nn"], a["B"], a["pt"], a["pts"], a["ps"],
                 a["phys"], a["vl"], a["up"], a["uq"], a["ul"], ws, 4096, None)
    assert sort(vl=None) == 1
    assert sort(up=None) == 1
    assert sort(ul=None) == 1
    assert sort(kb=8192) == 2
    assert sort(ps=12) == 2
    assert sort(B=0) == 0

    s = lib.dsa_sparse_mqa_logits_paired

    def sp(**kw):
        a = dict(kb=64, up=A16, uq=A16, ul=A16, vl=A16, ostride=512, nn=2)
        a.update(kw)
        return s(A16, A16, A16, A16, A16, 4, A16, 2, a["nn"], 32, 128, 64, 10, a["kb"], a["up"],
                 a["uq"], a["ul"], a["vl"], A16, 0, a["ostride"], ws, 4096, None)
    assert sp(vl=None) == 1
    assert sp(uq=None) == 1
    assert sp(kb=40) == 2
    assert sp(ostride=100) == 1
    assert sp(nn=5) == 2


def test_decode_step_rejects_before_launching(lib):
    """One-call decode step: a missing argument block, bad sizes and rows
    longer than one cluster launch takes are refused on the host, before any
    launch (the pointers are never dereferenced)."""
    import dsa_sparse_attention_paged_gb300 as D
    ws = ctypes.c_void_p(0x20000)
    assert lib.dsa_decode_step(None, ws, 4096, None) == 1

    def args(**kw):
        a = dict(q=0x10000, kv_pages=0x10000, kscale=0x10000, weights=0x10000,
                 page_table=0x10000, page_table_stride=4, context_lens=0x10000, B=2, next_n=1,
                 page_size=64, num_pages=10, k=2048, kb=512, logits=0x10000,
                 logits_stride=131072, histogram=0x10000, topk_idx=0x10000, block_ids=0x10000,
                 phys_blocks=0x10000, valid_lens=0x10000, sparse_scores=0x10000,
                 sparse_idx=0x10000)
        a.update(kw)
        return D.DecodeStepArgs(**a)
    assert lib.dsa_decode_step(ctypes.byref(args(kb=0)), ws, 4096, None) == 1
    assert lib.dsa_decode_step(ctypes.byref(args(next_n=0)), ws, 4096, None) == 1
    assert lib.dsa_decode_step(ctypes.byref(args(logits_stride=131080)), ws, 4096, None) == 2
    assert lib.dsa_decode_step(ctypes.byref(args(B=0)), ws, 4096, None) == 0
