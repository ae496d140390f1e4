"""Parity of the fused paged-MQA-logits + histogram kernel with the oracle,
through the C ABI.  Sizes span several 128-token tiles with ragged tails."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from tests.helpers import assert_close, live_mask, make, to_dev

pytestmark = pytest.mark.gpu

SENTINEL = -12345.0


def _run(case, stride, hist=None, ws=None):
    import dsa_sparse_attention_paged_gb300 as D
    d = to_dev(case)
    R = d["q"].shape[0]
    ws = ws or D.Workspace(R)
    logits = torch.full((R, stride), SENTINEL, dtype=torch.float32, device="cuda")
    D.paged_mqa_logits(d["q"], d["kv"], d["kscale"], d["weights"], d["page_table"],
                       d["context_lens"], case["next_n"], ws, logits=logits, histogram=hist)
    torch.cuda.synchronize()
    assert ws.status() == 0
    return logits.cpu().numpy()


CASES = [
    # (B, next_n, ctx lens, page size)
    (1, 1, [8192], 64),
    (3, 1, [1, 129, 1000], 64),
    (4, 1, [127, 128, 255, 4097], 128),
    (2, 2, [300, 513], 64),
    (3, 3, [130, 64, 2049], 64),
    (2, 4, [3, 1500], 64),
    (2, 4, [700, 129], 128),
    (5, 1, [0, 77, 0, 3000, 1], 64),
]


@pytest.mark.parametrize("B,nn,ctx,ps", CASES)
def test_logits_match_oracle_and_dead_columns_untouched(B, nn, ctx, ps):
    case = make(B, nn, ctx, ps, "normal", seed=100 + B * 10 + nn)
    stride = max(ctx) + 37
    got = _run(case, stride)
    ref = O.paged_mqa_logits(case["q"], case["kv"], case["kscale"], case["weights"],
                             case["page_table"], case["context_lens"], nn, ps,
                             logits_stride=stride, fill=np.nan)
    live, _ = live_mask(case["context_lens"], nn, stride)
    assert_close(got[live], ref[live], "logits")
    assert (got[~live] == SENTINEL).all(), "dead columns were written"


@pytest.mark.parametrize("nn,ps", [(1, 64), (2, 128), (4, 64)])
def test_integer_exact_case_is_bitwise(nn, ps):
    ctx = [2000, 333]
    case = make(2, nn, ctx, ps, "intexact", seed=7 + nn)
    got = _run(case, max(ctx))
    ref = O.paged_mqa_logits(case["q"], case["kv"], case["kscale"], case["weights"],
                             case["page_table"], case["context_lens"], nn, ps, fill=np.nan)
    live, _ = live_mask(case["context_lens"], nn, max(ctx))
    np.testing.assert_array_equal(got[live], ref[live])
    # the integer case lands on unit-bin edges, including negative integers
    assert (np.abs(ref[live]) >= 16).any() and (ref[live] <= -16).any()


@pytest.mark.parametrize("B,nn,ctx,ps,dist", [
    (3, 1, [1000, 4097, 5], 64, "mixed"),
    (2, 2, [2000, 130], 128, "unit"),
    (2, 4, [1025, 3000], 64, "fine"),
    (2, 3, [2048, 700], 64, "mixed"),
    (2, 1, [3000, 1500], 64, "intexact"),
])
def test_histogram_bitwise_on_own_logits_and_logits_unchanged(B, nn, ctx, ps, dist):
    import dsa_sparse_attention_paged_gb300 as D
    case = make(B, nn, ctx, ps, dist, seed=31 + nn)
    stride = max(ctx)
    R = B * nn
    plain = _run(case, stride)
    hist = torch.zeros((R, 1024), dtype=torch.int32, device="cuda")
    with_h = _run(case, stride, hist=hist)
    live, rl = live_mask(case["context_lens"], nn, stride)
    # logits bitwise identical with and without the histogram
    np.testing.assert_array_equal(plain[live], with_h[live])
    h = hist.cpu().numpy()
    ref = O.histogram(np.where(live, with_h, np.nan).astype(np.float32), rl)
    np.testing.assert_array_equal(h, ref)
    assert (h.sum(1) == rl).all()
    # counts accumulate across calls
    _run(case, stride, hist=hist)
    _run(case, stride, hist=hist)
    np.testing.assert_array_equal(hist.cpu().numpy(), 3 * ref)
    if dist == "mixed":
        b = np.argwhere(h.sum(0) > 0).ravel()
        assert b.min() == 0 or (h[:, :300].sum() > 0)  # the saturating/unit side is reached


def test_bad_page_id_is_flagged_not_faulted():
    import dsa_sparse_attention_paged_gb300 as D
    case = make(1, 1, [300], 64, "normal", seed=3)
    case["page_table"] = case["page_table"].copy()
    case["page_table"][0, 2] = case["num_pages"] + 100   # out of the pool
    d = to_dev(case)
    ws = D.Workspace(1)
    logits = torch.zeros((1, 300), dtype=torch.float32, device="cuda")
    D.paged_mqa_logits(d["q"], d["kv"], d["kscale"], d["weights"], d["page_table"],
                       d["context_lens"], 1, ws, logits=logits)
    torch.cuda.synchronize()
    assert ws.status() & D.DEV_BOUNDS
    ws.init()
    assert ws.status() == 0


@pytest.mark.parametrize("B,nn,ctx,ps,skip", [
    (3, 1, [4097, 9000, 130], 64, 0),
    (3, 1, [4097, 9000, 130], 64, 512),
    (2, 4, [3001, 700], 128, 64),
])
def test_fused_block_maxima_equal_block_amax8(B, nn, ctx, ps, skip):
    """Block maxima written by the logits kernel are bitwise those of
    dsa_block_amax8 on the same logits, and of the oracle."""
    import dsa_sparse_attention_paged_gb300 as D
    case = make(B, nn, ctx, ps, "mixed", seed=55 + skip)
    d = to_dev(case)
    R = B * nn
    stride = (max(ctx) + 7) // 8 * 8
    ws = D.Workspace(R)
    logits = torch.full((R, stride), float("nan"), dtype=torch.float32, device="cuda")
    fused = torch.full((R, stride // 8), -3.0, dtype=torch.float32, device="cuda")
    D.paged_mqa_logits(d["q"], d["kv"], d["kscale"], d["weights"], d["page_table"],
                       d["context_lens"], nn, ws, logits=logits, amax=fused,
                       amax_skip_if_blocks_le=skip)
    sep = torch.full((R, stride // 8), -3.0, dtype=torch.float32, device="cuda")
    D.block_amax8(logits, d["context_lens"], nn, ws, skip_if_blocks_le=skip, amax=sep)
    torch.cuda.synchronize()
    assert ws.status() == 0
    np.testing.assert_array_equal(fused.cpu().numpy(), sep.cpu().numpy())
    live, rl = live_mask(case["context_lens"], nn, stride)
    L = np.where(live, logits.cpu().numpy(), np.nan).astype(np.float32)
    ref = O.block_amax8(L, rl, skip_le=skip, amax_stride=stride // 8, fill=-3.0)
    np.testing.assert_array_equal(fused.cpu().numpy(), ref)


def test_histogram_counts_past_16_bits_per_slot():
    """One request of 80M keys (a 64-page pool referenced over and over): with
    q = 0 every score is +0, all in bin 511, so every histogram slot of every
    CTA counts far beyond 2^16 tokens of one bin; the periodic flush keeps the
    16-bit slot counts exact and the global count is the key count."""
    import dsa_sparse_attention_paged_gb300 as D
    n, ps, pool = 80_000_000, 64, 64
    npg = (n + ps - 1) // ps
    pt = (torch.arange(npg, dtype=torch.int32, device="cuda") % pool).reshape(1, npg)
    q = torch.zeros((1, 32, 128), dtype=torch.uint8, device="cuda")
    g = torch.Generator().manual_seed(12)
    kv = torch.randint(0, 256, (pool, ps, 128), generator=g, dtype=torch.uint8).cuda()
    kv[(kv & 0x7F) == 0x7F] = 0  # no NaN codes
    ks = torch.ones((pool, ps), dtype=torch.float32, device="cuda")
    w = torch.ones((1, 32), dtype=torch.float32, device="cuda")
    ctx = torch.tensor([n], dtype=torch.int32, device="cuda")
    hist = torch.zeros((1, 1024), dtype=torch.int32, device="cuda")
    ws = D.Workspace(1)
    L = D.paged_mqa_logits(q, kv, ks, w, pt, ctx, 1, ws, logits_stride=n, histogram=hist)
    torch.cuda.synchronize()
    assert ws.status() == 0
    assert bool((L == 0).all())
    h = hist.cpu().numpy()[0]
    assert h[511] == n and h.sum() == n
