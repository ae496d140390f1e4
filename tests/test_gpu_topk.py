"""Parity of the histogram-driven top-k (and its fallbacks) with the oracle's
full-sort top-k, computed on the GPU's own logits so the comparison is exact."""
import numpy as np
import pytest
import torch

import synthetic as S
from oracle import oracle as O
from tests.helpers import make, sets_equal, to_dev

pytestmark = pytest.mark.gpu


def _logits_and_hist(case, stride):
    import dsa_sparse_attention_paged_gb300 as D
    d = to_dev(case)
    R = d["q"].shape[0]
    ws = D.Workspace(R)
    logits = torch.full((R, stride), float("nan"), dtype=torch.float32, device="cuda")
    hist = torch.zeros((R, 1024), dtype=torch.int32, device="cuda")
    D.paged_mqa_logits(d["q"], d["kv"], d["kscale"], d["weights"], d["page_table"],
                       d["context_lens"], case["next_n"], ws, logits=logits, histogram=hist)
    return d, ws, logits, hist


@pytest.mark.parametrize("B,nn,ctx,ps,dist,k", [
    (2, 1, [8192, 5000], 64, "normal", 2048),
    (3, 1, [20000, 2047, 2049], 64, "mixed", 2048),
    (2, 4, [9000, 3000], 64, "unit", 2048),
    (2, 2, [4000, 700], 128, "fine", 512),
    (2, 1, [6000, 6000], 64, "intexact", 2048),   # heavy ties: lower column wins
    (1, 1, [100], 64, "normal", 2048),             # short row: -1 padding
    (3, 1, [0, 1, 5000], 64, "normal", 1),
])
def test_topk_matches_oracle(B, nn, ctx, ps, dist, k):
    import dsa_sparse_attention_paged_gb300 as D
    case = make(B, nn, ctx, ps, dist, seed=200 + k + nn)
    stride = max(ctx) + 8
    d, ws, logits, hist = _logits_and_hist(case, stride)
    R = B * nn
    flags = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    out = D.coarse_hist_topk(logits, d["context_lens"], nn, k, ws, histogram=hist,
                             reset_histogram=True, fallback_flags=flags)
    torch.cuda.synchronize()
    assert ws.status() == 0
    L = logits.cpu().numpy()
    ref = O.topk(L, O.row_lens(case["context_lens"], nn), k)
    assert sets_equal(out.cpu().numpy(), ref)
    assert (flags.cpu().numpy() == 0).all()
    assert (hist.cpu().numpy() == 0).all(), "reset_histogram left counts behind"


@pytest.mark.parametrize("longest", [12000, 20000])
def test_topk_without_histogram_builds_its_own(longest):
    """Rows that fit in shared memory take the one-CTA select; longer rows
    build their histogram in the workspace first."""
    import dsa_sparse_attention_paged_gb300 as D
    case = make(3, 1, [7000, longest, 300], 64, "mixed", seed=5)
    d, ws, logits, hist = _logits_and_hist(case, longest)
    out = D.coarse_hist_topk(logits, d["context_lens"], 1, 2048, ws, histogram=None)
    out2 = D.coarse_hist_topk(logits, d["context_lens"], 1, 2048, ws, histogram=None)
    torch.cuda.synchronize()
    ref = O.topk(logits.cpu().numpy(), O.row_lens(case["context_lens"], 1), 2048)
    assert sets_equal(out.cpu().numpy(), ref)
    assert sets_equal(out2.cpu().numpy(), ref)  # the workspace histogram was cleared


@pytest.mark.parametrize("kind", ["doubled", "zero", "shifted"])
def test_stale_histogram_falls_back_to_exact(kind):
    import dsa_sparse_attention_paged_gb300 as D
    case = make(2, 1, [9000, 4000], 64, "normal", seed=9)
    d, ws, logits, hist = _logits_and_hist(case, 9000)
    if kind == "doubled":
        hist *= 2
    elif kind == "zero":
        hist.zero_()
    else:
        hist.copy_(torch.roll(hist, 3, dims=1))
    flags = torch.zeros((2,), dtype=torch.int32, device="cuda")
    out = D.coarse_hist_topk(logits, d["context_lens"], 1, 2048, ws, histogram=hist,
                             fallback_flags=flags)
    torch.cuda.synchronize()
    ref = O.topk(logits.cpu().numpy(), O.row_lens(case["context_lens"], 1), 2048)
    assert sets_equal(out.cpu().numpy(), ref)
    f = flags.cpu().numpy()
    assert (f[0] == 1), f  # the long row must notice
    assert ws.status() == 0


def test_threshold_bin_over_capacity_falls_back_to_exact():
    """A flat region of 20000 equal scores makes bin T hold more than 8192
    candidates: the exact whole-row select takes over; ties -> lower column."""
    import dsa_sparse_attention_paged_gb300 as D
    R, n = 2, 30000
    x = S.random_logits(R, n, seed=4)
    x[:, 5000:25000] = 1.0
    x[1, 100] = np.nan
    L = torch.from_numpy(x).cuda()
    ctx = torch.full((R,), n, dtype=torch.int32, device="cuda")
    ws = D.Workspace(R)
    flags = torch.zeros((R,), dtype=torch.int32, device="cuda")
    out = D.coarse_hist_topk(L, ctx, 1, 2048, ws, histogram=None, fallback_flags=flags)
    torch.cuda.synchronize()
    ref = O.topk(x, np.full(R, n), 2048)
    assert sets_equal(out.cpu().numpy(), ref)
    assert (flags.cpu().numpy() == 2).all()


@pytest.mark.parametrize("n", [8192, 40000])
@pytest.mark.parametrize("c", [64, 65, 256, 257, 512])
def test_threshold_bin_sizes_around_the_rank_limits(n, c):
    """The threshold bin holds exactly c scores, of which the top 10 are taken
    (2038 scores lie in higher bins): up to 256 candidates are ranked in one
    pairwise pass, more by 1024-bin levels; rows of 8192 take the one-CTA
    select, rows of 40000 the cluster.  Row 0's candidates are distinct, row
    1's all equal (ties -> lower column)."""
    import dsa_sparse_attention_paged_gb300 as D
    k, above = 2048, 2038
    R = 2
    rng = np.random.default_rng(1000 + c + n)
    x = rng.uniform(-50.0, -10.0, (R, n)).astype(np.float32)
    cand_pos = []
    for r in range(R):
        pos = rng.permutation(n)
        x[r, pos[:above]] = rng.uniform(50.0, 100.0, above).astype(np.float32)
        cv = rng.uniform(1.001, 1.06, c) if r == 0 else np.full(c, 1.03125)
        x[r, pos[above:above + c]] = cv.astype(np.float32)
        cand_pos.append(pos[above:above + c])
    # the construction: the c candidates share one bin, and it is the bin the
    # 2048th score falls in
    for r in range(R):
        b = O.coarse_bins(x[r, cand_pos[r]])
        assert (b == b[0]).all()
        assert (O.coarse_bins(x[r]) == b[0]).sum() == c
    lens = np.full(R, n)
    hist = torch.from_numpy(O.histogram(x, lens)).cuda()
    L = torch.from_numpy(x).cuda()
    ctx = torch.full((R,), n, dtype=torch.int32, device="cuda")
    ws = D.Workspace(R)
    flags = torch.full((R,), 9, dtype=torch.int32, device="cuda")
    out = D.coarse_hist_topk(L, ctx, 1, k, ws, histogram=hist, fallback_flags=flags)
    torch.cuda.synchronize()
    assert sets_equal(out.cpu().numpy(), O.topk(x, lens, k))
    assert (flags.cpu().numpy() == 0).all(), flags
    assert ws.status() == 0


@pytest.mark.parametrize("lo,hi", [(223.0, 1000.0), (17.0, 17.9), (0.5, 0.53)])
def test_overflowing_bin_resolved_by_fine_histogram(lo, hi):
    """30000 distinct scores inside one coarse bin (the saturating bin, a unit
    bin, an FP16 bin): the histogram predicts the overflow, the fine pass
    resolves it exactly, no fallback."""
    import dsa_sparse_attention_paged_gb300 as D
    R, n = 3, 40000
    rng = np.random.default_rng(11)
    x = rng.normal(0, 1, (R, n)).astype(np.float32)
    x[:, 1000:31000] = rng.uniform(lo, hi, (R, 30000)).astype(np.float32)
    x[2, 5000:5100] = np.float32(lo)  # some exact ties as well
    L = torch.from_numpy(x).cuda()
    ctx = torch.full((R,), n, dtype=torch.int32, device="cuda")
    hist = torch.from_numpy(O.histogram(x, np.full(R, n))).cuda()
    ws = D.Workspace(R)
    flags = torch.full((R,), 9, dtype=torch.int32, device="cuda")
    for rep in range(2):
        out = D.coarse_hist_topk(L, ctx, 1, 2048, ws, histogram=hist, fallback_flags=flags)
        torch.cuda.synchronize()
        ref = O.topk(x, np.full(R, n), 2048)
        assert sets_equal(out.cpu().numpy(), ref), rep
        assert (flags.cpu().numpy() == 0).all(), flags
    assert ws.status() == 0


def test_nan_inf_and_short_rows():
    import dsa_sparse_attention_paged_gb300 as D
    R, n = 3, 5000
    x = S.random_logits(R, n, seed=6)
    x[0, ::7] = np.nan
    x[1, :10] = np.inf
    x[1, 10:20] = -np.inf
    x[2, :] = np.nan
    x[2, :1000] = -0.0
    x[2, 1000:1500] = 0.0
    L = torch.from_numpy(x).cuda()
    ctx = torch.tensor([n, n, n], dtype=torch.int32, device="cuda")
    ws = D.Workspace(R)
    for k in (1, 7, 2048):
        out = D.coarse_hist_topk(L, ctx, 1, k, ws, histogram=None)
        torch.cuda.synchronize()
        ref = O.topk(x, np.full(R, n), k)
        assert sets_equal(out.cpu().numpy(), ref), k


def test_len_div_rows_of_block_maxima():
    import dsa_sparse_attention_paged_gb300 as D
    R, n = 2, 4096
    x = S.random_logits(R, n, seed=8)
    L = torch.from_numpy(x).cuda()
    ctx = torch.tensor([8 * 4000 - 3, 8 * 700], dtype=torch.int32, device="cuda")
    ws = D.Workspace(R)
    out = D.coarse_hist_topk(L, ctx, 1, 512, ws, len_div=8)
    torch.cuda.synchronize()
    ref = O.topk(x, np.array([4000, 700]), 512)
    assert sets_equal(out.cpu().numpy(), ref)


@pytest.mark.parametrize("with_hist,overflow", [(True, False), (False, False), (True, True)])
def test_rows_longer_than_a_cluster_take_the_multi_cta_select(with_hist, overflow):
    """Rows over 131072 scores are split over many CTAs with global counters
    (and a fine pass when the threshold bin is over capacity)."""
    import dsa_sparse_attention_paged_gb300 as D
    R, n = 2, 150000
    rng = np.random.default_rng(21)
    x = rng.normal(0, 8, (R, n)).astype(np.float32)
    if overflow:
        x[:, 5000:45000] = rng.uniform(223.0, 900.0, (R, 40000)).astype(np.float32)
    L = torch.from_numpy(x).cuda()
    ctx = torch.full((R,), n, dtype=torch.int32, device="cuda")
    hist = torch.from_numpy(O.histogram(x, np.full(R, n))).cuda() if with_hist else None
    ws = D.Workspace(R)
    flags = torch.full((R,), 9, dtype=torch.int32, device="cuda")
    out = D.coarse_hist_topk(L, ctx, 1, 2048, ws, histogram=hist, fallback_flags=flags)
    torch.cuda.synchronize()
    ref = O.topk(x, np.full(R, n), 2048)
    assert sets_equal(out.cpu().numpy(), ref)
    assert (flags.cpu().numpy() == 0).all()
    assert ws.status() == 0
