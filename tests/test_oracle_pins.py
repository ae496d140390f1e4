"""Pins for the CPU oracle: each check ties the oracle to something other than
itself -- values derived by hand from the pages' rules (tests/golden), library
routines it does not use (torch / numpy FP8 and FP16 casts, torch.topk), closed
forms on constructed inputs, exhaustive sweeps and invariants.  A plausible
mistake (a dropped term, a wrong sign or index, a transposed operand, an
off-by-one bin constant) fails at least one of them.
"""
import math
import multiprocessing as mp
import os
import struct

import numpy as np
import pytest
import torch

from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32(h: int) -> float:
    return struct.unpack("<f", struct.pack("<I", h))[0]


# ---------------------------------------------------------------- O1: E4M3

def test_e4m3_table_matches_torch_cast_all_256_codes():
    tab = O.e4m3_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan_o, nan_r = np.isnan(tab), np.isnan(ref)
    assert (nan_o == nan_r).all()
    assert nan_o.sum() == 2  # S.1111.111
    np.testing.assert_array_equal(tab[~nan_o], ref[~nan_r])
    assert np.nanmax(tab) == 448.0 and np.nanmin(tab) == -448.0


# ---------------------------------------------------------------- FP16-RN

def _fp16_chunk(args):
    start, count = args
    from oracle import oracle as O2
    got = O2.fp16_rn_sweep(start, count)
    x = np.arange(start, start + count, dtype=np.uint64).astype(np.uint32).view(np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    isn = np.isnan(x)
    bad = (got != ref) & ~isn
    # NaN must stay NaN (payload is not specified)
    gh = got[isn]
    bad_nan = ~(((gh & 0x7C00) == 0x7C00) & ((gh & 0x3FF) != 0))
    return int(bad.sum()) + int(bad_nan.sum())


def test_fp16_rn_matches_numpy_cast_on_all_2pow32_patterns():
    """Exhaustive: the oracle's IEEE round-to-nearest-even binary16 conversion
    equals numpy's float32->float16 cast for every float32 bit pattern."""
    chunk = 1 << 26
    jobs = [(s, chunk) for s in range(0, 1 << 32, chunk)]
    ctx = mp.get_context("spawn")
    with ctx.Pool(min(8, os.cpu_count() or 1)) as pool:
        bad = sum(pool.map(_fp16_chunk, jobs))
    assert bad == 0


def _bf16_chunk(args):
    start, count = args
    import torch as T
    from oracle import oracle as O2
    got = O2.bf16_rn_sweep(start, count)
    u = np.arange(start, start + count, dtype=np.uint64).astype(np.uint32)
    x = u.view(np.float32)
    ref = T.from_numpy(x).to(T.bfloat16).view(T.int16).numpy().view(np.uint16)
    isn = np.isnan(x)
    bad = (got != ref) & ~isn
    gh = got[isn]
    bad_nan = ~(((gh & 0x7F80) == 0x7F80) & ((gh & 0x7F) != 0))
    return int(bad.sum()) + int(bad_nan.sum())


def test_bf16_rn_matches_torch_cast_on_all_2pow32_patterns():
    """Exhaustive: the oracle's bfloat16 round-to-nearest-even conversion
    (computed from the value) equals torch's float32->bfloat16 cast for every
    float32 bit pattern (NaN stays NaN)."""
    chunk = 1 << 26
    jobs = [(s, chunk) for s in range(0, 1 << 32, chunk)]
    ctx = mp.get_context("spawn")
    with ctx.Pool(min(8, os.cpu_count() or 1)) as pool:
        bad = sum(pool.map(_bf16_chunk, jobs))
    assert bad == 0


def test_bf16_decode_matches_torch_for_all_65536_codes():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    dec = np.array([O.bf16_bits_to_double(int(c)) for c in range(65536)])
    np.testing.assert_array_equal(np.isnan(dec), np.isnan(ref))
    ok = ~np.isnan(dec)
    np.testing.assert_array_equal(dec[ok], ref[ok])


# ---------------------------------------------------------------- O3: bins

def _golden_bins():
    rows = []
    with open(os.path.join(GOLDEN, "coarse_bins.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            h, _v, b = line.split()[:3]
            rows.append((int(h, 16), int(b)))
    return rows


def test_coarse_bin_golden_values():
    for h, b in _golden_bins():
        assert O.coarse_bin(f32(h)) == b, (hex(h), f32(h), b)


def test_coarse_bin_nan_is_not_counted():
    assert O.coarse_bin(float("nan")) == -1
    assert O.coarse_bin(f32(0xFFC00001)) == -1


def test_coarse_bin_unit_region_closed_form():
    # bin(n + f) = 511 - (304 + n - 16) = 223 - n and bin(-(n + f)) = 800 + n
    for n in range(16, 223):
        for frac in (0.0, 0.25, 0.5, 0.999):
            assert O.coarse_bin(n + frac) == 223 - n
            assert O.coarse_bin(-(n + frac)) == 800 + n


def test_coarse_bin_fine_region_matches_numpy_half_bits():
    # |x| < 16: bin = 511 - (half(|x|) >> 6) with numpy doing the rounding
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.uniform(-16, 16, 200000), rng.normal(0, 1e-3, 50000),
                        np.ldexp(1.0, np.arange(-30, 4))]).astype(np.float32)
    x = x[np.abs(x) < 16]
    m = (np.abs(x).astype(np.float16).view(np.uint16) >> 6).astype(np.int32)
    ref = np.where(np.signbit(x), 512 + m, 511 - m)
    np.testing.assert_array_equal(O.coarse_bins(x).astype(np.int32), ref)


def _bin_chunk(args):
    start, count = args
    from oracle import oracle as O2
    bins = O2.coarse_bin_sweep(start, count).astype(np.int32)
    pat = np.arange(start, start + count, dtype=np.uint64).astype(np.uint32)
    x = pat.view(np.float32)
    ok = ~np.isnan(x)
    b = bins[ok]
    # patterns increase -> |x| increases; positives: bins must not increase,
    # negatives: bins must not decrease
    if start < (1 << 31):
        mono = bool(np.all(np.diff(b) <= 0))
    else:
        mono = bool(np.all(np.diff(b) >= 0))
    nan_ok = bool(np.all(bins[~ok] == -1))
    present = np.zeros(1024, dtype=bool)
    present[np.unique(b)] = True
    first = int(b[0]) if b.size else None
    last = int(b[-1]) if b.size else None
    return mono, nan_ok, present, first, last


def test_coarse_bin_monotone_and_onto_all_2pow32_patterns():
    """Exhaustive: larger value -> bin index never larger; NaN never binned;
    every one of the 1024 bins is reachable."""
    chunk = 1 << 26
    jobs = [(s, chunk) for s in range(0, 1 << 32, chunk)]
    ctx = mp.get_context("spawn")
    with ctx.Pool(min(8, os.cpu_count() or 1)) as pool:
        res = pool.map(_bin_chunk, jobs)
    assert all(r[0] for r in res)
    assert all(r[1] for r in res)
    present = np.logical_or.reduce([r[2] for r in res])
    assert present.all()
    # chunk seams keep the order within each sign
    half = len(jobs) // 2
    for i in range(1, len(jobs)):
        if i == half or res[i][3] is None or res[i - 1][4] is None:
            continue
        if i < half:
            assert res[i][3] <= res[i - 1][4]
        else:
            assert res[i][3] >= res[i - 1][4]
    assert O.coarse_bin(-0.0) == O.coarse_bin(0.0) + 1


# ---------------------------------------------------------------- O2: logits

E4M3_ONE = 0x38  # 1.0
E4M3 = {v: int(torch.tensor([v]).to(torch.float8_e4m3fn).view(torch.uint8)) for v in
        [-4.0, -3.0, -2.0, -1.0, 0.0, 1.0, 2.0, 3.0, 4.0, 0.5, -0.5]}


def _case(B, nn, ctx, ps, H=32, D=128, seed=0):
    rng = np.random.default_rng(seed)
    pages = [(c + ps - 1) // ps for c in ctx]
    P = sum(pages) + 2
    perm = rng.permutation(P).astype(np.int32)
    pt = np.full((B, max(pages)), -1, np.int32)
    o = 0
    for b, n in enumerate(pages):
        pt[b, :n] = perm[o:o + n]
        o += n
    return P, pt


def _slot_to_token(pt, ps, B, ctx):
    m = {}
    for b in range(B):
        for t in range(ctx[b]):
            m[int(pt[b, t // ps]) * ps + t % ps] = (b, t)
    return m


def test_logits_closed_form_all_ones_query():
    """q = 1 everywhere, K row of token t = c_t everywhere:
    logit = sum_h w_h * ReLU(128 * c_t * kscale_t) -- checks the sum over d,
    the kscale product, ReLU and the head weighting."""
    B, nn, ps, H, D = 2, 1, 64, 32, 128
    ctx = [150, 77]
    P, pt = _case(B, nn, ctx, ps)
    rng = np.random.default_rng(1)
    vals = [-2.0, -1.0, 0.0, 1.0, 2.0, 3.0]
    cslot = rng.choice(vals, size=(P, ps))
    kv = np.vectorize(lambda v: E4M3[v])(cslot).astype(np.uint8)[:, :, None].repeat(D, axis=2)
    kscale = rng.uniform(0.5, 1.5, (P, ps)).astype(np.float32)
    q = np.full((B * nn, H, D), E4M3_ONE, np.uint8)
    w = rng.normal(0, 1, (B * nn, H)).astype(np.float32)
    L = O.paged_mqa_logits(q, kv, kscale, w, pt, np.array(ctx, np.int32), nn, ps)
    for b in range(B):
        for t in range(ctx[b]):
            slot = pt[b, t // ps] * ps + t % ps
            v = 128.0 * cslot.reshape(-1)[slot] * float(kscale.reshape(-1)[slot])
            v = max(v, 0.0)
            ref = np.float32(sum(float(x) * v for x in w[b]))
            assert L[b, t] == pytest.approx(ref, rel=1e-6, abs=1e-6)


def test_logits_closed_form_one_hot_heads_and_gather():
    """q[r,h] is a one-hot at d = (7h + 3r) % D with value s_h, and K of
    logical token t holds g(t, d) = ((t + 5d) % 7) - 3.  Then
    dot_h = s_h * g(t, d_h): a transposed operand, a wrong head/row index or a
    wrong page gather changes the result."""
    B, nn, ps, H, D = 2, 2, 64, 32, 128
    ctx = [200, 131]
    P, pt = _case(B, nn, ctx, ps, seed=3)
    slot_tok = _slot_to_token(pt, ps, B, ctx)
    kv = np.full((P, ps, D), E4M3[0.0], np.uint8)
    for slot, (b, t) in slot_tok.items():
        for d in range(D):
            kv.reshape(-1, D)[slot, d] = E4M3[float(((t + 5 * d) % 7) - 3)]
    kscale = np.full((P, ps), 0.5, np.float32)
    R = B * nn
    q = np.full((R, H, D), E4M3[0.0], np.uint8)
    s = np.array([[[1.0, 2.0, -1.0, 0.5][(h + r) % 4] for h in range(H)] for r in range(R)])
    for r in range(R):
        for h in range(H):
            q[r, h, (7 * h + 3 * r) % D] = E4M3[s[r, h]]
    w = np.array([[(h % 5) - 2 + 0.25 * r for h in range(H)] for r in range(R)], np.float32)
    L = O.paged_mqa_logits(q, kv, kscale, w, pt, np.array(ctx, np.int32), nn, ps)
    for r in range(R):
        b, j = divmod(r, nn)
        n_r = ctx[b] - (nn - 1 - j)
        for t in range(n_r):
            acc = 0.0
            for h in range(H):
                g = ((t + 5 * ((7 * h + 3 * r) % D)) % 7) - 3
                acc += float(w[r, h]) * max(s[r, h] * g * 0.5, 0.0)
            assert L[r, t] == np.float32(acc), (r, t)


def test_logits_next_n_rows_see_L_plus_j_keys():
    """Token j of a request sees L + j keys (DeepGEMM PR #94, "Producer cost"):
    with C = L + next_n - 1 the rows have L, L+1, ..., L+next_n-1 live columns."""
    B, nn, ps, L0 = 2, 4, 64, 100
    ctx = [L0 + nn - 1, 2 * L0 + nn - 1]
    P, pt = _case(B, nn, ctx, ps, seed=4)
    rng = np.random.default_rng(4)
    kv = rng.integers(0, 0x70, (P, ps, 128)).astype(np.uint8)
    q = rng.integers(0, 0x70, (B * nn, 32, 128)).astype(np.uint8)
    w = rng.normal(0, 1, (B * nn, 32)).astype(np.float32)
    ks = np.ones((P, ps), np.float32)
    out = O.paged_mqa_logits(q, kv, ks, w, pt, np.array(ctx, np.int32), nn, ps,
                             logits_stride=max(ctx) + 5, fill=np.nan)
    for b in range(B):
        for j in range(nn):
            live = ~np.isnan(out[b * nn + j])
            assert live.sum() == ctx[b] - (nn - 1 - j)
            assert live[:ctx[b] - (nn - 1 - j)].all()
    np.testing.assert_array_equal(O.row_lens(ctx, nn),
                                  [L0, L0 + 1, L0 + 2, L0 + 3, 2 * L0, 2 * L0 + 1, 2 * L0 + 2,
                                   2 * L0 + 3])


def test_logits_at_matches_dense():
    import synthetic as S
    w = S.Workload("t", 2, 2, [300, 171], 64, "normal", 11)
    d = S.generate(w)
    L = O.paged_mqa_logits(d["q"], d["kv"], d["kscale"], d["weights"], d["page_table"],
                           d["context_lens"], 2, 64)
    rows = np.array([0, 1, 2, 3, 3], np.int64)
    cols = np.array([0, 298, 5, 170, 169], np.int64)
    v = O.logits_at(d["q"], d["kv"], d["kscale"], d["weights"], d["page_table"], 2, 64, rows, cols)
    np.testing.assert_array_equal(v, L[rows, cols])


# ---------------------------------------------------------------- histogram

def test_histogram_counts_live_non_nan_and_accumulates():
    x = np.array([[1.0, np.nan, -1.0, 300.0, 16.0, 7.0, np.nan, 5.0],
                  [0.0, -0.0, np.inf, -np.inf, 2.0, 2.0, 2.0, 9.0]], np.float32)
    rl = np.array([6, 7], np.int64)  # row 0: 6 live (one NaN), row 1: 7 live
    h = O.histogram(x, rl)
    assert h[0].sum() == 5 and h[1].sum() == 7
    assert h[0, 271] == 1 and h[0, 752] == 1 and h[0, 0] == 1 and h[0, 207] == 1
    assert h[1, 511] == 1 and h[1, 512] == 1 and h[1, 0] == 1 and h[1, 1023] == 1
    assert h[1, O.coarse_bin(2.0)] == 3
    h3 = O.histogram(x, rl, O.histogram(x, rl, h))
    np.testing.assert_array_equal(h3, 3 * h)


# ---------------------------------------------------------------- O4: top-k

def _is_topk(row, n, k, sel):
    """The defining property, checked pairwise: every selected entry beats every
    unselected live non-NaN entry under (value desc, column asc)."""
    live = [t for t in range(n) if not math.isnan(row[t])]
    s = [t for t in sel if t >= 0]
    if len(s) != min(k, len(live)) or len(set(s)) != len(s):
        return False
    rest = set(live) - set(s)

    def key(t):
        u = struct.unpack("<I", struct.pack("<f", float(row[t])))[0]
        return (u ^ 0xFFFFFFFF) if u & 0x80000000 else (u | 0x80000000)

    for a in s:
        for b in rest:
            if not (key(a) > key(b) or (key(a) == key(b) and a < b)):
                return False
    return all(t == -1 for t in sel[len(s):])


def test_topk_brute_force_tiny_rows():
    rng = np.random.default_rng(7)
    for trial in range(300):
        n = int(rng.integers(0, 14))
        k = int(rng.integers(1, 9))
        row = rng.choice([-2.0, -1.0, -0.0, 0.0, 0.5, 1.0, 3.0, np.inf, -np.inf, np.nan],
                         size=max(n, 1)).astype(np.float32)
        out = O.topk(row[None, :], np.array([n]), k)[0]
        assert _is_topk(row, n, k, list(out)), (row[:n], k, out)


def test_topk_distinct_rows_match_torch_topk():
    g = torch.Generator().manual_seed(3)
    x = torch.randn(4, 5000, generator=g)
    x = x + torch.arange(5000) * 1e-3  # distinct
    out = O.topk(x.numpy(), np.full(4, 5000), 300)
    ref = torch.topk(x, 300, dim=1).indices.numpy()
    for r in range(4):
        assert set(out[r].tolist()) == set(ref[r].tolist())


def test_topk_all_equal_takes_lowest_columns_and_pads():
    row = np.zeros((1, 100), np.float32)
    out = O.topk(row, np.array([100]), 10)[0]
    assert out.tolist() == list(range(10))
    out = O.topk(row, np.array([7]), 10)[0]
    assert out.tolist() == list(range(7)) + [-1] * 3


# ---------------------------------------------------------------- O5/O6

def test_amax8_closed_form_on_arange_rows():
    n = [1, 8, 9, 64, 77]
    x = np.tile(np.arange(80, dtype=np.float32), (len(n), 1))
    a = O.block_amax8(x, np.array(n), skip_le=0, amax_stride=12, fill=-7.0)
    for r, nr in enumerate(n):
        nb = (nr + 7) // 8
        for i in range(12):
            if i < nb - 1:
                assert a[r, i] == 8 * i + 7
            elif i == nb - 1:
                assert a[r, i] == np.inf
            else:
                assert a[r, i] == -7.0  # nothing past the count
    a = O.block_amax8(x, np.array(n), skip_le=8, amax_stride=12, fill=-7.0)
    assert (a[:4] == -7.0).all() and a[4, 9] == np.inf  # nb = 1, 1, 2, 8 skipped; 10 kept


def test_amax8_nan_and_signed_zero_handling():
    x = np.array([[np.nan, 1.0, np.nan, -3.0, 0, 0, 0, 0] + [np.nan] * 8 +
                  [-0.0, 0.0, -0.0, -1.0, -0.0, -2.0, -0.0, -0.0] +
                  [-0.0, -0.0, -5.0, -0.0, -0.0, -0.0, -0.0, -0.0] + [1.0]], np.float32)
    a = O.block_amax8(x, np.array([33]), amax_stride=5)
    assert a[0, 0] == 1.0 and np.isnan(a[0, 1]) and a[0, 4] == np.inf
    assert a[0, 2] == 0.0 and not np.signbit(a[0, 2])  # +0 is above -0
    assert a[0, 3] == 0.0 and np.signbit(a[0, 3])


def test_block_table_closed_form():
    """amax[i] = (37 i) mod nb for nb = 1000 (a permutation: distinct values);
    the top kb = 100 blocks are the newest (+inf) and those with value >= 901
    other than the newest; identity for short rows; physical block and live
    length from the page table and row lengths."""
    nb, kb, ps = 1000, 100, 64
    n_long = 8 * nb - 3  # newest block holds 5 live tokens
    n_short = 8 * 60 - 1
    rl = np.array([n_long, n_short], np.int64)
    amax = np.zeros((2, nb), np.float32)
    amax[0] = (37 * np.arange(nb)) % nb
    amax[0, nb - 1] = np.inf
    pages = (n_long + ps - 1) // ps
    pt = np.stack([np.arange(pages)[::-1], np.arange(pages) + 1000]).astype(np.int32)
    table, phys, vl = O.block_table(amax, rl, np.array([0, 1], np.int32), kb, pt, ps)
    vals = (37 * np.arange(nb - 1)) % nb
    want = sorted([int(i) for i in np.argsort(-vals, kind="stable")[:kb - 1]] + [nb - 1])
    assert table[0].tolist() == want
    assert table[1, :60].tolist() == list(range(60)) and (table[1, 60:] == 2**31 - 1).all()
    for r in range(2):
        for i in range(kb):
            bid = table[r, i]
            if bid == 2**31 - 1:
                assert phys[r, i] == 2**31 - 1
                continue
            tok = 8 * bid
            assert phys[r, i] == (pt[r, tok // ps] * ps + tok % ps) // 8
    assert vl[0] == 8 * (kb - 1) + 5 and vl[1] == n_short


def test_sparse_logits_closed_form_positions_and_mask():
    """K of logical token t holds c(t) = (t % 5) - 2 at d = 0 and 0 elsewhere; q =
    one-hot at d = 0 with value 1: logit(t) = sum_h w_h ReLU(c(t) * ks)."""
    B, ps, D, H = 1, 64, 128, 32
    ctx = [333]
    P, pt = _case(B, 1, ctx, ps, seed=9)
    kv = np.full((P, ps, D), E4M3[0.0], np.uint8)
    for slot, (b, t) in _slot_to_token(pt, ps, B, ctx).items():
        kv.reshape(-1, D)[slot, 0] = E4M3[float((t % 5) - 2)]
    q = np.full((1, H, D), E4M3[0.0], np.uint8)
    q[0, :, 0] = E4M3_ONE
    w = np.linspace(-1, 2, H).astype(np.float32)
    ks = np.full((P, ps), 2.0, np.float32)
    table = np.array([[3, 10, 41, 2**31 - 1]], np.int32)  # block 41 holds tokens 328..335
    out = O.sparse_logits(q, kv, ks, w, pt, np.array([333]), np.array([0], np.int32), ps, table)
    for i in range(32):
        bid = table[0, i // 8]
        t = int(bid) * 8 + i % 8
        if bid == 2**31 - 1 or t >= 333:
            assert out[0, i] == -np.inf
        else:
            v = max(((t % 5) - 2) * 2.0, 0.0)
            assert out[0, i] == np.float32(sum(float(x) * v for x in w))


# ---------------------------------------------------------------- O8

def test_fp16_order_matches_numpy_over_all_65536_encodings():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = codes.view(np.float16)
    nonnan = ~np.isnan(vals)
    k = int(nonnan.sum())
    out = O.topk_fp16(codes[None, :], np.array([65536], np.int32), k)[0]
    sel_vals = vals[out].astype(np.float64)
    assert np.all(np.diff(sel_vals) <= 0)  # non-increasing values
    assert sorted(out.tolist()) == np.nonzero(nonnan)[0].tolist()  # every non-NaN once
    # +0 ranks above -0 (sign bit decides), equal keys never occur otherwise
    assert out.tolist().index(0x0000) < out.tolist().index(0x8000)
    # and the half decode matches numpy for every code
    dec = np.array([O.fp16_bits_to_double(int(c)) for c in range(0, 65536, 17)])
    np.testing.assert_array_equal(np.isnan(dec), np.isnan(vals[::17].astype(np.float64)))
    ok = ~np.isnan(dec)
    np.testing.assert_array_equal(dec[ok], vals[::17].astype(np.float64)[ok])


def test_bf16_order_matches_torch_over_all_65536_encodings():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nonnan = ~np.isnan(vals)
    k = int(nonnan.sum())
    out = O.topk_bf16(codes[None, :], np.array([65536], np.int32), k)[0]
    assert np.all(np.diff(vals[out]) <= 0)  # non-increasing values
    assert sorted(out.tolist()) == np.nonzero(nonnan)[0].tolist()  # every non-NaN once
    assert out.tolist().index(0x0000) < out.tolist().index(0x8000)  # +0 above -0
    # a BF16 NaN is not an FP16 NaN (and the other way round): the formats'
    # own rules decide
    assert 0x7C01 in out.tolist() and 0x7F81 not in out.tolist()


def test_bf16_topk_ties_to_lower_position_and_table_mapping():
    one5 = int(torch.tensor([1.5]).to(torch.bfloat16).view(torch.int16).item()) & 0xFFFF
    two = int(torch.tensor([2.0]).to(torch.bfloat16).view(torch.int16).item()) & 0xFFFF
    s = np.full((1, 40), one5, np.uint16)
    s[0, 33] = two
    s[0, 5] = 0x7FC0  # NaN
    table = np.array([[4, 9, 13, 20, 21]], np.int32)
    out = O.topk_bf16(s, np.array([37], np.int32), 5, table)[0]
    pos = [33, 0, 1, 2, 3]
    assert out.tolist() == [table[0, p // 8] * 8 + p % 8 for p in pos]
    out = O.topk_bf16(s, np.array([7], np.int32), 8)[0]
    assert out.tolist() == [0, 1, 2, 3, 4, 6, -1, -1]


def test_fp16_topk_ties_to_lower_position_and_table_mapping():
    s = np.full((1, 40), np.float16(1.5)).view(np.uint16)
    s[0, 33] = np.float16(2.0).view(np.uint16)
    table = np.array([[4, 9, 13, 20, 21]], np.int32)
    out = O.topk_fp16(s, np.array([37], np.int32), 5, table)[0]
    pos = [33, 0, 1, 2, 3]
    assert out.tolist() == [table[0, p // 8] * 8 + p % 8 for p in pos]
    out = O.topk_fp16(s, np.array([3], np.int32), 5)[0]
    assert out.tolist() == [0, 1, 2, -1, -1]


IMAX = 2**31 - 1


def _pad(ids, kb):
    return list(ids) + [IMAX] * (kb - len(ids))


def test_pair_union_worked_example():
    """Two rows of one request, tables [1 4 7] and [2 4 9 11] (kb = 4): the
    union is [1 2 4 7 9 11]; block 4 is held by both rows (A at 1, B at 1)."""
    kb = 4
    table = np.array([_pad([1, 4, 7], kb), _pad([2, 4, 9, 11], kb)], np.int32)
    phys = np.where(table == IMAX, IMAX, table + 100).astype(np.int32)
    up, uq, ul = O.pair_union(table, phys, 2)
    assert ul.tolist() == [6]
    assert up[0, :6].tolist() == [101, 102, 104, 107, 109, 111]
    pos_a = (uq[0, :6] & 0xFFFF) - 1
    pos_b = (uq[0, :6] >> 16) - 1
    assert pos_a.tolist() == [0, -1, 1, 2, -1, -1]
    assert pos_b.tolist() == [-1, 0, 1, -1, 2, 3]
    assert (up[0, 6:] == IMAX).all() and (uq[0, 6:] == 0).all()


@pytest.mark.parametrize("next_n", [1, 2, 3, 4, 5])
def test_pair_union_brute_force_by_sets(next_n):
    """Against Python sets on random tiny tables: units are rows (2m, 2m+1) of
    a request, an odd last row alone; every union entry is a block of one of
    the two rows, in ascending order, with each row's own table position."""
    rng = np.random.default_rng(7 + next_n)
    B, kb = 3, 6
    R = B * next_n
    table = np.full((R, kb), IMAX, np.int32)
    for r in range(R):
        n = int(rng.integers(0, kb + 1))
        table[r, :n] = np.sort(rng.choice(14, size=n, replace=False))
    phys = np.where(table == IMAX, IMAX, 1000 + 3 * table + (np.arange(R)[:, None] // next_n))
    phys = phys.astype(np.int32)
    up, uq, ul = O.pair_union(table, phys, next_n)
    upr = (next_n + 1) // 2
    assert up.shape == (B * upr, 2 * kb)
    for u in range(B * upr):
        b, m = divmod(u, upr)
        ra = b * next_n + 2 * m
        rows = [ra] + ([ra + 1] if 2 * m + 1 < next_n else [])
        lists = [[int(x) for x in table[r] if x != IMAX] for r in rows]
        want = sorted(set().union(*map(set, lists)))
        assert ul[u] == len(want)
        for e, blk in enumerate(want):
            assert up[u, e] == 1000 + 3 * blk + b
            for j, lst in enumerate(lists):
                got = int((uq[u, e] >> (16 * j)) & 0xFFFF) - 1
                assert got == (lst.index(blk) if blk in lst else -1)
            if len(rows) == 1:
                assert uq[u, e] >> 16 == 0
        assert (up[u, len(want):] == IMAX).all() and (uq[u, len(want):] == 0).all()


def test_pair_union_covers_each_row_position_once():
    """Invariant: over a unit's union, each row's positions 0..n-1 appear
    exactly once (the pass writes every live slot of both rows once)."""
    rng = np.random.default_rng(11)
    kb, R = 64, 8
    table = np.full((R, kb), IMAX, np.int32)
    for r in range(R):
        n = int(rng.integers(kb // 2, kb + 1))
        table[r, :n] = np.sort(rng.choice(200, size=n, replace=False))
    up, uq, ul = O.pair_union(table, table, 4)
    for u in range(len(ul)):
        for j in range(2):
            r = (u // 2) * 4 + 2 * (u % 2) + j
            n = int((table[r] != IMAX).sum())
            pos = ((uq[u, :ul[u]] >> (16 * j)) & 0xFFFF).astype(np.int64) - 1
            assert sorted(pos[pos >= 0].tolist()) == list(range(n))


def test_ue8m0_matches_torch_for_all_256_codes():
    """UE8M0 block exponents against torch's float8_e8m0fnu decode: 2^(e-127),
    255 is NaN."""
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = np.array([O.ue8m0(e) for e in range(256)])
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])


def test_e2m1_matches_torch_e4m3_through_the_exponent_rebias():
    """Every E2M1 code decodes to the E4M3 value with the same sign, the
    exponent field moved from bias 1 to bias 7 and the mantissa bit on top
    (the subnormal 0.5 becomes the normal 2^-1): the direct E2M1 -> E4M3
    unpacking the pages name, checked against torch's E4M3 decode."""
    def rebias(c):
        s, e, m = c >> 3, (c >> 1) & 3, c & 1
        if e == 0:
            bits = 0 if m == 0 else (6 << 3)
        else:
            bits = ((e + 6) << 3) | (m << 2)
        return (s << 7) | bits
    e4 = torch.tensor([rebias(c) for c in range(16)], dtype=torch.uint8)
    ref = e4.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([O.e2m1(c) for c in range(16)])
    np.testing.assert_array_equal(got, ref)
    np.testing.assert_array_equal(np.signbit(got), np.signbit(ref))
    assert got.max() == 6.0 and sorted(set(np.abs(got)))[1] == 0.5  # largest, smallest step


def _pack_mx(vals, exps):
    """[slots][128] E2M1 codes -> [slots][64] bytes (even dimension in the low
    nibble) and [slots][4] block exponents (already codes)."""
    codes = np.asarray(vals, np.uint8)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8), np.asarray(exps, np.uint8)


def test_mx_logits_closed_form_uniform_keys():
    """q = 1 everywhere, every key element 1.0 (code 2) with all four block
    exponents e_t: logit = sum_h w_h * 128 * 2^(e_t - 127)."""
    B, nn, ps, H, D = 2, 1, 64, 32, 128
    ctx = [150, 77]
    P, pt = _case(B, nn, ctx, ps, seed=5)
    rng = np.random.default_rng(2)
    e_slot = rng.integers(120, 135, size=P * ps)
    codes, exps = _pack_mx(np.full((P * ps, D), 2), np.repeat(e_slot[:, None], 4, axis=1))
    q = np.full((B * nn, H, D), E4M3_ONE, np.uint8)
    w = rng.normal(0, 1, (B * nn, H)).astype(np.float32)
    L = O.paged_mqa_logits_mx(q, codes.reshape(P, ps, 64), exps.reshape(P, ps, 4), w, pt,
                              np.array(ctx, np.int32), nn, ps)
    for b in range(B):
        for t in range(ctx[b]):
            slot = pt[b, t // ps] * ps + t % ps
            v = 128.0 * 2.0 ** (int(e_slot[slot]) - 127)
            assert L[b, t] == np.float32(sum(float(x) * v for x in w[b]))
        assert np.isnan(L[b, ctx[b]:]).all()


def test_mx_logits_nibble_order_and_block_exponents():
    """q[r,h] one-hot at d_h = (9h + 5r) % 128 (even and odd dimensions, all
    four blocks); key element d of logical token t has code c(t, d) in
    1..15 and block b of token t exponent 125 + (t + b) % 5.  Then
    dot_h = E2M1(c(t, d_h)) * 2^(e(t, d_h / 32) - 127): a swapped nibble, a
    wrong block index or a wrong page gather changes the result."""
    B, nn, ps, H, D = 2, 2, 64, 32, 128
    ctx = [140, 99]
    P, pt = _case(B, nn, ctx, ps, seed=9)
    val = np.zeros((P * ps, D), np.uint8)
    ex = np.full((P * ps, 4), 127, np.uint8)
    code = lambda t, d: 1 + (3 * t + 7 * d) % 15
    for slot, (b, t) in _slot_to_token(pt, ps, B, ctx).items():
        val[slot] = [code(t, d) for d in range(D)]
        ex[slot] = [125 + (t + k) % 5 for k in range(4)]
    codes, exps = _pack_mx(val, ex)
    R = B * nn
    q = np.full((R, H, D), E4M3[0.0], np.uint8)
    s = np.array([[[1.0, 2.0, -1.0, 0.5][(h + r) % 4] for h in range(H)] for r in range(R)])
    for r in range(R):
        for h in range(H):
            q[r, h, (9 * h + 5 * r) % D] = E4M3[s[r, h]]
    w = np.array([[(h % 5) - 2 + 0.25 * r for h in range(H)] for r in range(R)], np.float32)
    L = O.paged_mqa_logits_mx(q, codes.reshape(P, ps, 64), exps.reshape(P, ps, 4), w, pt,
                              np.array(ctx, np.int32), nn, ps)
    mag = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for r in range(R):
        b, j = divmod(r, nn)
        for t in range(ctx[b] - (nn - 1 - j)):
            acc = 0.0
            for h in range(H):
                d = (9 * h + 5 * r) % D
                c = code(t, d)
                k = (-1 if c & 8 else 1) * mag[c & 7] * 2.0 ** ((t + d // 32) % 5 - 2)
                acc += float(w[r, h]) * max(s[r, h] * k, 0.0)
            assert L[r, t] == np.float32(acc), (r, t)


def test_mx_logits_equal_fp8_logits_when_block_exponents_agree():
    """A key whose four block exponents equal e is the E4M3 key of the same
    elements (E2M1 -> E4M3 by the exponent rebias) with kscale 2^(e - 127);
    both oracles are exact in double up to the final rounding, so the MXFP4
    logits equal the FP8 logits bit for bit (ties O10 to the pinned O2)."""
    def rebias(c):
        s, e, m = c >> 3, (c >> 1) & 3, c & 1
        return (s << 7) | ((6 << 3) if (e == 0 and m) else 0 if e == 0 else ((e + 6) << 3) | (m << 2))
    B, nn, ps, H, D = 2, 2, 64, 32, 128
    ctx = [300, 170]
    P, pt = _case(B, nn, ctx, ps, seed=21)
    rng = np.random.default_rng(21)
    val = rng.integers(0, 16, size=(P * ps, D))
    e_slot = rng.integers(118, 136, size=P * ps)
    codes, exps = _pack_mx(val, np.repeat(e_slot[:, None], 4, axis=1))
    kv = np.vectorize(rebias)(val).astype(np.uint8).reshape(P, ps, D)
    kscale = np.ldexp(1.0, e_slot - 127).astype(np.float32).reshape(P, ps)
    finite = [c for c in range(256) if (c & 0x7F) != 0x7F]
    q = rng.choice(finite, size=(B * nn, H, D)).astype(np.uint8)
    w = rng.normal(0, 1, (B * nn, H)).astype(np.float32)
    c = np.array(ctx, np.int32)
    L_mx = O.paged_mqa_logits_mx(q, codes.reshape(P, ps, 64), exps.reshape(P, ps, 4), w, pt, c,
                                 nn, ps)
    L_f8 = O.paged_mqa_logits(q, kv, kscale, w, pt, c, nn, ps)
    np.testing.assert_array_equal(L_mx.view(np.uint32), L_f8.view(np.uint32))


def test_mx_logits_at_matches_dense_mx_logits():
    """The sampled MXFP4 logits (used for full-size checks) equal the dense
    ones at the same (row, column), on a seeded MXFP4 workload."""
    import synthetic as S
    w = S.Workload("mx small", 3, 2, [700, 65, 1300], 64, "normal", 77, key_format="mxfp4")
    c = S.generate(w)
    L = O.paged_mqa_logits_mx(c["q"], c["k_codes"], c["k_exp"], c["weights"], c["page_table"],
                              c["context_lens"], 2, 64)
    rl = O.row_lens(c["context_lens"], 2)
    rng = np.random.default_rng(3)
    rows = rng.integers(0, 6, 500)
    cols = (rng.random(500) * rl[rows]).astype(np.int64)
    got = O.logits_at_mx(c["q"], c["k_codes"], c["k_exp"], c["weights"], c["page_table"], 2, 64,
                         rows, cols)
    np.testing.assert_array_equal(got, L[rows, cols])
    assert c["k_codes"].shape == (c["num_pages"], 64, 64) and c["k_exp"].shape[-1] == 4
    # the FP8 inputs of the seed do not move when MXFP4 keys are drawn too
    f8 = S.generate(S.Workload("mx small", 3, 2, [700, 65, 1300], 64, "normal", 77))
    for k in ("q", "kv", "kscale", "weights", "page_table"):
        np.testing.assert_array_equal(f8[k], c[k])
