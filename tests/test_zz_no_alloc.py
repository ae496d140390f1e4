"""The allocation-free top-k entry point (for callers that cannot allocate a
workspace) gives the same results as the workspace entry point, on two calls
in a row, through the C ABI.  Collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _case():
    import synthetic as S
    from tests.helpers import make, to_dev
    import dsa_sparse_attention_paged_gb300 as D
    case = make(4, 1, [20000, 9000, 130, 16000], 64, "mixed", seed=606)
    d = to_dev(case)
    ws = D.Workspace(4)
    stride = 20008
    logits = torch.full((4, stride), float("nan"), dtype=torch.float32, device="cuda")
    hist = torch.zeros((4, 1024), dtype=torch.int32, device="cuda")
    D.paged_mqa_logits(d["q"], d["kv"], d["kscale"], d["weights"], d["page_table"],
                       d["context_lens"], 1, ws, logits=logits, histogram=hist)
    torch.cuda.synchronize()
    return D, d, ws, logits, hist


def _sorted(t):
    return np.sort(t.cpu().numpy(), axis=1)


def test_noalloc_topk_matches_workspace_topk_twice():
    D, d, ws, logits, hist = _case()
    ctx = d["context_lens"]
    ref = D.coarse_hist_topk(logits, ctx, 1, 2048, ws, histogram=hist)
    ref_nohist = D.coarse_hist_topk(logits, ctx, 1, 2048, ws, histogram=None)
    torch.cuda.synchronize()
    for call in range(2):
        flags = torch.full((4,), -1, dtype=torch.int32, device="cuda")
        out = torch.full((4, 2048), -7, dtype=torch.int32, device="cuda")
        st = D.lib.dsa_coarse_hist_topk_noalloc(
            ctypes.c_void_p(logits.data_ptr()), logits.stride(0), ctypes.c_void_p(ctx.data_ptr()),
            1, 1, 4, ctypes.c_void_p(hist.data_ptr()), 0, 2048,
            ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(flags.data_ptr()),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 0, D.lib.dsa_status_string(st)
        out2 = D.coarse_hist_topk_noalloc(logits, ctx, 1, 2048, histogram=None)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(_sorted(out), _sorted(ref))
        np.testing.assert_array_equal(_sorted(out2), _sorted(ref_nohist))
        assert (flags.cpu().numpy() >= 0).all()


def test_noalloc_short_rows_without_histogram():
    import dsa_sparse_attention_paged_gb300 as D
    from oracle import oracle as O
    rng = np.random.default_rng(8)
    x = rng.normal(0, 5, (3, 9000)).astype(np.float32)
    L = torch.from_numpy(x).cuda()
    ctx = torch.tensor([8 * 9000 - 5, 8 * 700, 8 * 4000], dtype=torch.int32, device="cuda")
    for call in range(2):
        out = D.coarse_hist_topk_noalloc(L, ctx, 1, 512, len_div=8)
        torch.cuda.synchronize()
        ref = O.topk(x, np.array([9000, 700, 4000]), 512)
        np.testing.assert_array_equal(_sorted(out), np.sort(ref, axis=1))


def test_noalloc_rejects_rows_beyond_its_maximum():
    import dsa_sparse_attention_paged_gb300 as D
    n = D.NOALLOC_MAX_ROWS + 1
    x = torch.zeros((n, 64), dtype=torch.float32, device="cuda")
    c = torch.full((n,), 64, dtype=torch.int32, device="cuda")
    o = torch.zeros((n, 8), dtype=torch.int32, device="cuda")
    st = D.lib.dsa_coarse_hist_topk_noalloc(
        ctypes.c_void_p(x.data_ptr()), 64, ctypes.c_void_p(c.data_ptr()), 1, 1, n, None, 0, 8,
        ctypes.c_void_p(o.data_ptr()), None, None)
    assert st == 2  # DSA_ERR_UNSUPPORTED


def _overcap_rows(R, n, rng):
    """Rows whose threshold bin holds more than the candidate capacity: many
    equal scores (the exact whole-row fallback, flag 2), many distinct scores
    inside one coarse bin (the fine histogram, flag 0), plain rows, short
    rows (k or fewer scores: every score taken)."""
    x = rng.uniform(-60.0, 0.0, (R, n)).astype(np.float32)
    for r in range(R):
        big = rng.permutation(n)[:1000 + 100 * r]
        x[r, big] = rng.uniform(100.0, 200.0, big.size).astype(np.float32)
        rest = np.setdiff1d(np.arange(n), big)
        pos = rng.permutation(rest)[:20000]
        if r % 3 == 0:
            x[r, pos] = 5.0                                    # one key: ties
        elif r % 3 == 1:
            x[r, pos] = rng.uniform(5.0, 5.2, pos.size).astype(np.float32)  # one coarse bin
    return x


def test_noalloc_over_capacity_bins_then_fewer_rows():
    import dsa_sparse_attention_paged_gb300 as D
    from oracle import oracle as O
    rng = np.random.default_rng(99)
    R, n, k = 8, 40000, 2048
    x = _overcap_rows(R, n, rng)
    ctx_h = np.array([40000, 40000, 40000, 30000, 2000, 40000, 35000, 1], np.int32)
    hist_h = O.histogram(x, ctx_h.astype(np.int64))
    ref = O.topk(x, ctx_h.astype(np.int64), k)
    L = torch.from_numpy(x).cuda()
    ctx = torch.from_numpy(ctx_h).cuda()
    hist = torch.from_numpy(hist_h).cuda()
    ws = D.Workspace(R)
    wflags = torch.full((R,), -1, dtype=torch.int32, device="cuda")
    wout = D.coarse_hist_topk(L, ctx, 1, k, ws, histogram=hist, fallback_flags=wflags)
    torch.cuda.synchronize()
    wf = wflags.cpu().numpy()
    assert (wf[[0, 3, 6]] == 2).all() and (wf[[1, 4, 7]] == 0).all(), wf
    np.testing.assert_array_equal(_sorted(wout), np.sort(ref, axis=1))
    for rows in (R, 2):  # a call on fewer rows after one on more: stale rows stay out
        flags = torch.full((R,), -1, dtype=torch.int32, device="cuda")
        out = torch.full((R, k), -7, dtype=torch.int32, device="cuda")
        D.coarse_hist_topk_noalloc(L, ctx, 1, k, histogram=hist, out=out, fallback_flags=flags,
                                   R=rows)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(flags.cpu().numpy()[:rows], wf[:rows])
        assert (flags.cpu().numpy()[rows:] == -1).all()
        np.testing.assert_array_equal(_sorted(out[:rows]), np.sort(ref[:rows], axis=1))
        assert (out[rows:].cpu().numpy() == -7).all()
        # the caller's histogram is read, not changed, without reset_histogram
        np.testing.assert_array_equal(hist.cpu().numpy(), hist_h)
