"""The batched select (several independent top-k problems, one launch) and
the windowed fine histogram of the two widest coarse bins, against the
oracle's full-sort top-k on the same scores."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from tests.helpers import make, sets_equal, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,nn,ctx,ps,dist", [
    (3, 1, [40000, 9000, 70000], 64, "mixed"),     # logits rows: clusters; maxima: one CTA a row
    (2, 2, [131072, 20000], 64, "normal"),         # the longest rows a cluster takes
    (9, 1, [5000] * 4 + [16000] * 5, 64, "unit"),  # short rows only: eight rows a cluster
])
def test_logits_and_block_maxima_in_one_launch(B, nn, ctx, ps, dist):
    import dsa_sparse_attention_paged_gb300 as D
    case = make(B, nn, ctx, ps, dist, seed=300 + B)
    d = to_dev(case)
    R = B * nn
    stride = (max(ctx) + 7) // 8 * 8
    ws = D.Workspace(2 * R)
    logits = torch.full((R, stride), float("nan"), dtype=torch.float32, device="cuda")
    hist = torch.zeros((R, 1024), dtype=torch.int32, device="cuda")
    amax = torch.full((R, stride // 8), float("nan"), dtype=torch.float32, device="cuda")
    D.paged_mqa_logits(d["q"], d["kv"], d["kscale"], d["weights"], d["page_table"],
                       d["context_lens"], nn, ws, logits=logits, histogram=hist, amax=amax)
    flags = torch.full((2, R), 9, dtype=torch.int32, device="cuda")
    outs = D.coarse_hist_topk_batch([
        dict(logits=logits, context_lens=d["context_lens"], next_n=nn, k=2048, histogram=hist,
             reset_histogram=True, fallback_flags=flags[0]),
        dict(logits=amax, context_lens=d["context_lens"], next_n=nn, k=512, len_div=8,
             fallback_flags=flags[1])], ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    rl = O.row_lens(case["context_lens"], nn)
    L = logits.cpu().numpy()
    assert sets_equal(outs[0].cpu().numpy(), O.topk(L, rl, 2048))
    A = amax.cpu().numpy()
    assert sets_equal(outs[1].cpu().numpy(), O.topk(A, (rl + 7) // 8, 512))
    assert (flags.cpu().numpy() == 0).all()
    assert (hist.cpu().numpy() == 0).all()
    # the workspace is left zeroed: a second batch on it gives the same result
    hist2 = torch.from_numpy(O.histogram(L, rl)).cuda()
    again = D.coarse_hist_topk_batch([
        dict(logits=logits, context_lens=d["context_lens"], next_n=nn, k=2048, histogram=hist2),
        dict(logits=amax, context_lens=d["context_lens"], next_n=nn, k=512, len_div=8)], ws)
    torch.cuda.synchronize()
    assert sets_equal(again[0].cpu().numpy(), outs[0].cpu().numpy())
    assert sets_equal(again[1].cpu().numpy(), outs[1].cpu().numpy())


def test_batch_with_a_long_row_problem_runs_in_sequence_and_skips_empty():
    import dsa_sparse_attention_paged_gb300 as D
    rng = np.random.default_rng(5)
    x1 = rng.normal(0, 4, (2, 150000)).astype(np.float32)   # longer than a cluster's row
    x2 = rng.normal(0, 4, (3, 3000)).astype(np.float32)
    ctx1 = torch.full((2,), 150000, dtype=torch.int32, device="cuda")
    ctx2 = torch.tensor([3000, 17, 2500], dtype=torch.int32, device="cuda")
    L1, L2 = torch.from_numpy(x1).cuda(), torch.from_numpy(x2).cuda()
    empty = torch.zeros((0, 64), dtype=torch.float32, device="cuda")
    ws = D.Workspace(5)
    o1, o0, o2 = D.coarse_hist_topk_batch([
        dict(logits=L1, context_lens=ctx1, next_n=1, k=2048),
        dict(logits=empty, context_lens=ctx2, next_n=1, k=16),
        dict(logits=L2, context_lens=ctx2, next_n=1, k=100)], ws)
    torch.cuda.synchronize()
    assert ws.status() == 0 and o0.shape == (0, 16)
    assert sets_equal(o1.cpu().numpy(), O.topk(x1, np.full(2, 150000), 2048))
    assert sets_equal(o2.cpu().numpy(), O.topk(x2, np.array([3000, 17, 2500]), 100))


def test_batch_rejects_a_small_workspace_before_launching():
    import dsa_sparse_attention_paged_gb300 as D
    x = torch.zeros((4, 100), dtype=torch.float32, device="cuda")
    ctx = torch.full((4,), 100, dtype=torch.int32, device="cuda")
    ws = D.Workspace(6)
    with pytest.raises(D.DSAError) as e:
        D.coarse_hist_topk_batch([dict(logits=x, context_lens=ctx, next_n=1, k=8)] * 2, ws)
    assert e.value.status == 5


@pytest.mark.parametrize("n", [40000, 12000])
@pytest.mark.parametrize("kind", ["pos_saturating", "neg_saturating", "tiny"])
def test_widest_bins_use_a_fine_window(kind, n):
    """Bin T is |x| >= 223 or |x| below the smallest FP16 step, whose key
    ranges are far wider than the fine histogram: the window at the end nearer
    to magnitude 1 is resolved, keys beyond it clamp to the end fine bins;
    the result stays exact (clusters at n = 40000, one CTA at n = 12000)."""
    import dsa_sparse_attention_paged_gb300 as D
    R = 3
    rng = np.random.default_rng(17)
    x = rng.normal(-50, 1, (R, n)).astype(np.float32)
    m = 6000
    if kind == "pos_saturating":
        x[:, :m] = np.exp(rng.uniform(np.log(223.0), np.log(1e9), (R, m))).astype(np.float32)
        x[1, :3000] = np.exp(rng.uniform(np.log(1e6), np.log(1e30), 3000)).astype(np.float32)
    elif kind == "neg_saturating":
        x = -np.exp(rng.uniform(np.log(223.0), np.log(1e12), (R, n))).astype(np.float32)
        x[2, :50] = -np.inf
    else:
        x[:, :m] = rng.uniform(0, 3.5e-6, (R, m)).astype(np.float32)
        x[1, :2000] = rng.uniform(0, 1e-30, 2000).astype(np.float32)
        x[2, :100] = 0.0
    L = torch.from_numpy(x).cuda()
    ctx = torch.full((R,), n, dtype=torch.int32, device="cuda")
    hist = torch.from_numpy(O.histogram(x, np.full(R, n))).cuda()
    ws = D.Workspace(R)
    for h in (hist, None):
        out = D.coarse_hist_topk(L, ctx, 1, 2048, ws, histogram=h)
        torch.cuda.synchronize()
        assert ws.status() == 0
        assert sets_equal(out.cpu().numpy(), O.topk(x, np.full(R, n), 2048)), h is None


def _block_ref(L, rl, kb):
    nb = (rl + 7) // 8
    A = O.block_amax8(L, rl, skip_le=0, amax_stride=(L.shape[1] + 7) // 8)
    return O.topk(A, nb, kb)


@pytest.mark.parametrize("B,nn,ctx,ps,dist,kb", [
    (3, 1, [40000, 9000, 70000], 64, "mixed", 512),  # clusters, ragged last blocks
    (2, 2, [131072, 20001], 64, "normal", 512),      # the longest rows a cluster takes
    (9, 1, [5000] * 4 + [16000] * 5, 64, "unit", 512),  # one CTA a row
    (2, 3, [3000, 100000], 128, "fine", 2048),       # block_k = k, short rows take all
    (3, 1, [7, 4097, 0], 64, "normal", 16),          # tiny and empty rows
])
def test_fused_block_maxima_select(B, nn, ctx, ps, dist, kb):
    """Top-kb of the block maxima chosen in the same launch as the top-2048
    of the scores: the same sets as block_amax8 + top-k over the maxima."""
    import dsa_sparse_attention_paged_gb300 as D
    case = make(B, nn, ctx, ps, dist, seed=400 + B + kb)
    d = to_dev(case)
    R = B * nn
    stride = (max(ctx) + 7) // 8 * 8 or 8
    ws = D.Workspace(R)
    logits = torch.full((R, stride), float("nan"), dtype=torch.float32, device="cuda")
    hist = torch.zeros((R, 1024), dtype=torch.int32, device="cuda")
    D.paged_mqa_logits(d["q"], d["kv"], d["kscale"], d["weights"], d["page_table"],
                       d["context_lens"], nn, ws, logits=logits, histogram=hist)
    flags = torch.full((2, R), 9, dtype=torch.int32, device="cuda")
    (out, bout), = D.coarse_hist_topk_batch([
        dict(logits=logits, context_lens=d["context_lens"], next_n=nn, k=2048, histogram=hist,
             reset_histogram=True, fallback_flags=flags[0], block_k=kb,
             block_fallback_flags=flags[1])], ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    rl = O.row_lens(case["context_lens"], nn)
    L = logits.cpu().numpy()
    assert sets_equal(out.cpu().numpy(), O.topk(L, rl, 2048))
    assert sets_equal(bout.cpu().numpy(), _block_ref(L, rl, kb))
    assert (flags.cpu().numpy() == 0).all(), flags


@pytest.mark.parametrize("table", [False, True])
@pytest.mark.parametrize("n", [60000, 12000])
@pytest.mark.parametrize("kind", ["nan_blocks", "tied_maxima", "wide_bin", "inf_blocks",
                                  "plain"])
def test_fused_block_select_edge_cases(kind, n, table):
    """All-NaN blocks are never chosen; thousands of equal maxima overflow the
    candidate slots and take the exact fallback (ties to the lower block);
    maxima spread over the saturating bin use the fine window; more blocks at
    +inf than the table holds take the lowest of them.  With `table` the
    block output is the sorted block table (written by the whole cluster in
    the plain case), checked with its physical blocks and live lengths."""
    import dsa_sparse_attention_paged_gb300 as D
    R = 3
    rng = np.random.default_rng(23)
    x = rng.normal(0, 2, (R, n)).astype(np.float32)
    if kind == "nan_blocks":
        x[:, : n // 2] = np.nan
        x[1, 8 * 100: 8 * 101 - 3] = 5.0     # a block with a few NaN still counts
    elif kind == "tied_maxima":
        x[:, :] = rng.normal(-5, 1, (R, n)).astype(np.float32)
        x[:, ::8] = 1.0                      # every block has the same maximum
    elif kind == "wide_bin":
        x[:, ::3] = np.exp(rng.uniform(np.log(223.0), np.log(1e7), (R, (n + 2) // 3)))
    elif kind == "inf_blocks":
        x[:, 8 * 37: 8 * 37 + 8 * 700: 8] = np.inf  # 700 blocks at +inf (rows of 12000: fewer)
    L = torch.from_numpy(x).cuda()
    ctx = torch.tensor([n, n - 5, n // 3], dtype=torch.int32, device="cuda")
    hist = torch.from_numpy(O.histogram(x, ctx.cpu().numpy())).cuda()
    ws = D.Workspace(R)
    bflags = torch.full((R,), 9, dtype=torch.int32, device="cuda")
    ps = 64
    extra = {}
    if table:
        # each row its own request; pages of a request a permutation of a pool
        npg = (n + ps - 1) // ps
        pt_h = np.stack([rng.permutation(R * npg)[:npg] for _ in range(R)]).astype(np.int32)
        phys = torch.full((R, 512), -5, dtype=torch.int32, device="cuda")
        vlen = torch.full((R,), -5, dtype=torch.int32, device="cuda")
        extra = dict(block_page_table=torch.from_numpy(pt_h).cuda(), block_page_size=ps,
                     block_phys=phys, block_valid_lens=vlen)
    (out, bout), = D.coarse_hist_topk_batch([
        dict(logits=L, context_lens=ctx, next_n=1, k=2048, histogram=hist, block_k=512,
             block_fallback_flags=bflags, **extra)], ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    rl = ctx.cpu().numpy().astype(np.int64)
    assert sets_equal(out.cpu().numpy(), O.topk(x, rl, 2048))
    ids, ref = bout.cpu().numpy(), _block_ref(x, rl, 512)
    if table:
        # the table pads with INT32_MAX, and a row of at most 512 blocks takes
        # the identity table (checked against the oracle's table below)
        ids = np.where(ids == np.iinfo(np.int32).max, -1, ids)
        big = (rl + 7) // 8 > 512
        ids, ref = ids[big], ref[big]
    assert sets_equal(ids, ref)
    f = bflags.cpu().numpy()
    assert set(f.tolist()) <= ({0, 2} if kind == "tied_maxima" else {0}), f
    if table:
        A = O.block_amax8(x, rl, skip_le=512, amax_stride=(n + 7) // 8, fill=0.0)
        t_ref, p_ref, v_ref = O.block_table(A, rl, np.arange(R, dtype=np.int32), 512, pt_h, ps)
        np.testing.assert_array_equal(bout.cpu().numpy(), t_ref)
        np.testing.assert_array_equal(phys.cpu().numpy(), p_ref)
        np.testing.assert_array_equal(vlen.cpu().numpy(), v_ref)


@pytest.mark.parametrize("B,nn,ctx,ps", [
    (3, 1, [40000, 3000, 131072], 64),   # a short row takes the identity table
    (2, 2, [70001, 9000], 128),
    (4, 1, [16000, 20000, 4097, 100000], 64),
])
def test_select_writes_sorted_block_table(B, nn, ctx, ps):
    """The block output written as the sorted block table in the select
    launch equals the separate sort_candidate_blocks of the same ids: table,
    physical blocks and live lengths, bitwise; NaN-only blocks in a short row
    still take their identity slot."""
    import dsa_sparse_attention_paged_gb300 as D
    case = make(B, nn, ctx, ps, "normal", seed=800 + B)
    d = to_dev(case)
    R = B * nn
    kb = 512
    stride = (max(ctx) + 7) // 8 * 8
    ws = D.Workspace(R)
    logits = torch.full((R, stride), float("nan"), dtype=torch.float32, device="cuda")
    hist = torch.zeros((R, 1024), dtype=torch.int32, device="cuda")
    D.paged_mqa_logits(d["q"], d["kv"], d["kscale"], d["weights"], d["page_table"],
                       d["context_lens"], nn, ws, logits=logits, histogram=hist)
    rl = O.row_lens(case["context_lens"], nn)
    short = int(np.argmin(rl))
    logits[short, 8:40] = float("nan")  # NaN-only blocks 1..4 of the shortest row
    hist2 = torch.from_numpy(O.histogram(logits.cpu().numpy(), rl)).cuda()
    outs = []
    for fused in (False, True):
        table = torch.full((R, kb), -5, dtype=torch.int32, device="cuda")
        phys = torch.full((R, kb), -5, dtype=torch.int32, device="cuda")
        vlen = torch.full((R,), -5, dtype=torch.int32, device="cuda")
        extra = dict(block_page_table=d["page_table"], block_page_size=ps, block_phys=phys,
                     block_valid_lens=vlen) if fused else {}
        D.coarse_hist_topk_batch([dict(logits=logits, context_lens=d["context_lens"], next_n=nn,
                                       k=2048, histogram=hist2.clone(), block_k=kb,
                                       block_out=table, **extra)], ws)
        if not fused:
            D.sort_candidate_blocks(table, d["context_lens"], nn, d["page_table"], ps, ws,
                                    phys_blocks=phys, valid_lens=vlen)
        torch.cuda.synchronize()
        assert ws.status() == 0
        outs.append([t.cpu().numpy() for t in (table, phys, vlen)])
    for a, b in zip(*outs):
        np.testing.assert_array_equal(a, b)
    A = O.block_amax8(logits.cpu().numpy(), rl, skip_le=kb, amax_stride=(stride + 7) // 8,
                      fill=0.0)
    t_ref, p_ref, v_ref = O.block_table(A, rl, np.arange(R, dtype=np.int32) // nn, kb,
                                        case["page_table"], ps)
    np.testing.assert_array_equal(outs[1][0], t_ref)
    np.testing.assert_array_equal(outs[1][1], p_ref)
    np.testing.assert_array_equal(outs[1][2], v_ref)


@pytest.mark.parametrize("R", [48, 47])
@pytest.mark.parametrize("given_hist", [True, False])
def test_two_rows_a_cluster(R, given_hist):
    """More rows of at most 65536 scores than one wave of row clusters holds
    (more than 38 on 152 SMs): an even count goes two rows to a cluster, four
    CTAs each, an odd count one row a cluster.  The row mix puts the two rows
    of a cluster on different paths: a row of k or fewer scores beside a full
    one, an empty row, rows that end inside the first CTA's slice, rows whose
    threshold bin needs the fine histogram.  Top-k sets, the sorted block
    table, its physical blocks and live lengths against the oracle; the
    workspace is left zeroed (a second run gives the same result)."""
    import dsa_sparse_attention_paged_gb300 as D
    rng = np.random.default_rng(900 + R + 2 * given_hist)
    n, ps, kb = 65536, 64, 512
    x = rng.normal(0, 2, (R, n)).astype(np.float32)
    narrow = np.arange(1, R, 4)  # one coarse bin holds almost the whole row
    x[narrow] = (1.0 + rng.uniform(0.0, 0.06, (len(narrow), n))).astype(np.float32)
    lens = rng.integers(16385, n + 1, R)
    lens[[0, 2, 3, 5, 6, 7, 9, 10]] = [n, 2048, 0, 100, 2049, 16000, n - 3, 4096]
    lens[R - 1] = 12001
    ctx = torch.from_numpy(lens.astype(np.int32)).cuda()
    L = torch.from_numpy(x).cuda()
    npg = n // ps
    pt_h = np.stack([rng.permutation(2 * npg)[:npg] for _ in range(R)]).astype(np.int32)
    ws = D.Workspace(R)
    res = []
    for _ in range(2):
        table = torch.full((R, kb), -5, dtype=torch.int32, device="cuda")
        phys = torch.full((R, kb), -5, dtype=torch.int32, device="cuda")
        vlen = torch.full((R,), -5, dtype=torch.int32, device="cuda")
        hist = torch.from_numpy(O.histogram(x, lens)).cuda() if given_hist else None
        ((out, _),) = D.coarse_hist_topk_batch([
            dict(logits=L, context_lens=ctx, next_n=1, k=2048, histogram=hist, block_k=kb,
                 block_out=table, block_page_table=torch.from_numpy(pt_h).cuda(),
                 block_page_size=ps, block_phys=phys, block_valid_lens=vlen)], ws)
        torch.cuda.synchronize()
        assert ws.status() == 0
        res.append([t.cpu().numpy() for t in (out, table, phys, vlen)])
    rl = lens.astype(np.int64)
    assert sets_equal(res[0][0], O.topk(x, rl, 2048))
    A = O.block_amax8(x, rl, skip_le=kb, amax_stride=n // 8, fill=0.0)
    t_ref, p_ref, v_ref = O.block_table(A, rl, np.arange(R, dtype=np.int32), kb, pt_h, ps)
    np.testing.assert_array_equal(res[0][1], t_ref)
    np.testing.assert_array_equal(res[0][2], p_ref)
    np.testing.assert_array_equal(res[0][3], v_ref)
    assert sets_equal(res[1][0], res[0][0])
    for a, b in zip(res[0][1:], res[1][1:]):
        np.testing.assert_array_equal(a, b)
