"""Parity of the two-level candidate path with the oracle: block amax8, block
top-k, the ascending padded block table, sparse logits (bitwise equal to the
dense logits at the chosen positions) and the FP16 packed top-k."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from tests.helpers import assert_close, make, sets_equal, to_dev

pytestmark = pytest.mark.gpu
IMAX = 2**31 - 1


def _dense(case, stride):
    import dsa_sparse_attention_paged_gb300 as D
    d = to_dev(case)
    R = d["q"].shape[0]
    ws = D.Workspace(R)
    logits = torch.full((R, stride), float("nan"), dtype=torch.float32, device="cuda")
    D.paged_mqa_logits(d["q"], d["kv"], d["kscale"], d["weights"], d["page_table"],
                       d["context_lens"], case["next_n"], ws, logits=logits)
    return d, ws, logits


@pytest.mark.parametrize("ctx,kb,ps,nn", [
    ([40000, 3000, 20001], 512, 128, 1),
    ([9000, 17], 256, 64, 1),
    ([12000, 5000], 512, 64, 2),
])
def test_two_level_chain(ctx, kb, ps, nn):
    import dsa_sparse_attention_paged_gb300 as D
    B = len(ctx)
    R = B * nn
    case = make(B, nn, ctx, ps, "normal", seed=400 + kb)
    stride = max(ctx) + 16
    d, ws, logits = _dense(case, stride)
    rl = O.row_lens(case["context_lens"], nn)
    L = logits.cpu().numpy()

    # amax8 (rows with nb <= kb skipped)
    amax_stride = (stride + 7) // 8
    amax = torch.full((R, amax_stride), -5.0, dtype=torch.float32, device="cuda")
    D.block_amax8(logits, d["context_lens"], nn, ws, skip_if_blocks_le=kb, amax=amax)
    A = amax.cpu().numpy()
    refA = O.block_amax8(L, rl, skip_le=kb, amax_stride=amax_stride, fill=-5.0)
    np.testing.assert_array_equal(A, refA)

    # block top-k on the GPU's amax, rows with nb > kb compared
    ids = D.coarse_hist_topk(amax, d["context_lens"], nn, kb, ws, len_div=8)
    nb = (rl + 7) // 8
    ref_ids = O.topk(A, nb, kb)
    got_ids = ids.cpu().numpy()
    for r in range(R):
        if nb[r] > kb:
            assert sets_equal(got_ids[r:r + 1], ref_ids[r:r + 1]), r

    # sort -> table, phys, valid lens
    phys = torch.empty((R, kb), dtype=torch.int32, device="cuda")
    vl = torch.empty((R,), dtype=torch.int32, device="cuda")
    D.sort_candidate_blocks(ids, d["context_lens"], nn, d["page_table"], ps, ws,
                            phys_blocks=phys, valid_lens=vl)
    rtr = np.arange(R, dtype=np.int32) // nn
    t_ref, p_ref, v_ref = O.block_table(A, rl, rtr, kb, case["page_table"], ps)
    np.testing.assert_array_equal(ids.cpu().numpy(), t_ref)
    np.testing.assert_array_equal(phys.cpu().numpy(), p_ref)
    np.testing.assert_array_equal(vl.cpu().numpy(), v_ref)

    # sparse logits: oracle tolerance, and bitwise equal to the dense logits
    sp = D.sparse_mqa_logits(d["q"], d["kv"], d["kscale"], d["weights"], d["page_table"],
                             d["context_lens"], nn, ids, ws, out_dtype=D.OUT_F32)
    sp16 = D.sparse_mqa_logits(d["q"], d["kv"], d["kscale"], d["weights"], d["page_table"],
                               d["context_lens"], nn, ids, ws, out_dtype=D.OUT_F16)
    torch.cuda.synchronize()
    assert ws.status() == 0
    SP = sp.cpu().numpy()
    ref_sp = O.sparse_logits(case["q"], case["kv"], case["kscale"], case["weights"],
                             case["page_table"], rl, rtr, ps, t_ref)
    masked = np.isneginf(ref_sp)
    np.testing.assert_array_equal(np.isneginf(SP), masked)
    assert_close(SP[~masked], ref_sp[~masked], "sparse logits")
    pos = np.arange(kb * 8)
    for r in range(R):
        tok = t_ref[r, pos // 8].astype(np.int64) * 8 + pos % 8
        ok = ~masked[r]
        np.testing.assert_array_equal(SP[r, ok], L[r, tok[ok]])
    # live positions are a prefix of length valid_len
    for r in range(R):
        assert (~masked[r, :v_ref[r]]).all() and masked[r, v_ref[r]:].all()
    # FP16 output is the RN-even rounding of the FP32 one
    np.testing.assert_array_equal(sp16.cpu().numpy().view(np.uint16), O.fp16_rn_array(SP))
    # reading the K rows through the sort's physical blocks and live lengths
    # gives bitwise the same scores, FP32 and FP16
    for dt, ref in ((D.OUT_F32, sp), (D.OUT_F16, sp16)):
        via = D.sparse_mqa_logits(d["q"], d["kv"], d["kscale"], d["weights"], d["page_table"],
                                  d["context_lens"], nn, ids, ws, out_dtype=dt,
                                  phys_blocks=phys, valid_lens=vl)
        torch.cuda.synchronize()
        assert torch.equal(via.view(torch.int16 if dt == D.OUT_F16 else torch.int32),
                           ref.view(torch.int16 if dt == D.OUT_F16 else torch.int32))

    # FP16 top-2048 with the fused table transform, on the GPU's own FP16 scores
    k = 2048
    top = D.topk_fp16(sp16, vl, k, ws, block_table=ids)
    torch.cuda.synchronize()
    ref_top = O.topk_fp16(sp16.cpu().numpy().view(np.uint16), v_ref, k, t_ref)
    assert sets_equal(top.cpu().numpy(), ref_top)

    # the BF16 sibling: RN-even of the FP32 scores, and its select
    spb = D.sparse_mqa_logits(d["q"], d["kv"], d["kscale"], d["weights"], d["page_table"],
                              d["context_lens"], nn, ids, ws, out_dtype=D.OUT_BF16,
                              phys_blocks=phys, valid_lens=vl)
    torch.cuda.synchronize()
    SB = spb.view(torch.int16).cpu().numpy().view(np.uint16)
    np.testing.assert_array_equal(SB, O.bf16_rn_array(SP))
    topb = D.topk_bf16(spb, vl, k, ws, block_table=ids)
    torch.cuda.synchronize()
    assert sets_equal(topb.cpu().numpy(), O.topk_bf16(SB, v_ref, k, t_ref))


def test_fp16_topk_ties_nan_and_positions():
    import dsa_sparse_attention_paged_gb300 as D
    rng = np.random.default_rng(3)
    R, n = 4, 6000
    vals = rng.normal(0, 4, (R, n)).astype(np.float16)
    vals[0, :] = np.float16(1.0)                      # all ties
    vals[1, ::3] = np.float16(np.nan)
    vals[2, :50] = np.float16(np.inf)
    vals[2, 50:60] = np.float16(-np.inf)
    vals[3, 100:200] = np.float16(-0.0)
    s = torch.from_numpy(vals.view(np.uint16).copy()).cuda()
    ws = D.Workspace(R)
    for vl_list, k in (([n, n, n, n], 2048), ([5999, 17, 2048, 1], 2048), ([n, 4001, 3, 0], 1)):
        vl = torch.tensor(vl_list, dtype=torch.int32, device="cuda")
        out = D.topk_fp16(s, vl, k, ws)
        torch.cuda.synchronize()
        ref = O.topk_fp16(vals.view(np.uint16), np.array(vl_list, np.int32), k)
        assert sets_equal(out.cpu().numpy(), ref), (vl_list, k)


def test_fp16_order_keys_all_65536_encodings():
    import dsa_sparse_attention_paged_gb300 as D
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    keys = D.fp16_order_keys(torch.from_numpy(codes.copy()).cuda()).cpu().numpy()
    vals = codes.view(np.float16).astype(np.float64)
    nan = np.isnan(vals)
    assert (keys[nan] == 0).all()
    kk = keys[~nan].astype(np.int64)
    v = vals[~nan]
    assert len(np.unique(kk)) == kk.size  # one key per encoding
    order = np.argsort(kk)
    assert np.all(np.diff(v[order]) >= 0)  # key order == value order
    # +0 above -0
    assert keys[0x0000] > keys[0x8000]
    assert (kk > 0).all()


def test_bf16_topk_ties_nan_and_positions():
    import dsa_sparse_attention_paged_gb300 as D
    rng = np.random.default_rng(4)
    R, n = 4, 6000
    vals = torch.from_numpy(rng.normal(0, 4, (R, n)).astype(np.float32))
    vals[0, :] = 1.0                       # all ties
    vals[1, ::3] = float("nan")
    vals[2, :50] = float("inf")
    vals[2, 50:60] = -float("inf")
    vals[3, 100:200] = -0.0
    bits = vals.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    bits[1, 1::7] = 0x7F81                 # a NaN pattern that is no NaN in FP16
    s = torch.from_numpy(bits).cuda()
    ws = D.Workspace(R)
    for vl_list, k in (([n, n, n, n], 2048), ([5999, 17, 2048, 1], 2048), ([n, 4001, 3, 0], 1)):
        vl = torch.tensor(vl_list, dtype=torch.int32, device="cuda")
        out = D.topk_bf16(s, vl, k, ws)
        torch.cuda.synchronize()
        ref = O.topk_bf16(bits, np.array(vl_list, np.int32), k)
        assert sets_equal(out.cpu().numpy(), ref), (vl_list, k)


def test_bf16_order_keys_all_65536_encodings():
    import dsa_sparse_attention_paged_gb300 as D
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    keys = D.bf16_order_keys(torch.from_numpy(codes.copy()).cuda()).cpu().numpy()
    vals = np.array([O.bf16_bits_to_double(int(c)) for c in codes])
    nan = np.isnan(vals)
    assert (keys[nan] == 0).all()
    kk = keys[~nan].astype(np.int64)
    v = vals[~nan]
    assert len(np.unique(kk)) == kk.size  # one key per encoding
    order = np.argsort(kk)
    assert np.all(np.diff(v[order]) >= 0)  # keys ascend with the value
    assert kk[np.nonzero(codes[~nan] == 0x8000)[0][0]] < kk[np.nonzero(codes[~nan] == 0)[0][0]]



def _verify_ids(ctx, nn, kb, seed):
    """Block ids per row in the shape the block top-k gives (any order, -1
    padded): rows with more than kb blocks take kb (or, for a few, fewer)
    distinct blocks including the newest; the second row of each pair shares
    most of the first one's blocks, as draft rows of one request do."""
    rng = np.random.default_rng(seed)
    rl = O.row_lens(np.asarray(ctx, np.int32), nn)
    R = len(rl)
    ids = np.full((R, kb), -1, np.int32)
    prev = None
    for r in range(R):
        nb = int((rl[r] + 7) // 8)
        if nb <= kb:
            ids[r, :] = rng.integers(-1, max(nb, 1), size=kb)  # ignored: identity table
            prev = None
            continue
        take = kb if rng.random() < 0.8 else int(rng.integers(1, kb))
        if prev is not None and r % nn % 2 == 1:
            keep = [x for x in prev if x < nb - 1][: int(0.7 * take)]
            rest = np.setdiff1d(np.arange(nb - 1), keep)
            extra = rng.choice(rest, size=take - 1 - len(keep), replace=False)
            chosen = np.concatenate([keep, extra, [nb - 1]]).astype(np.int32)
        else:
            chosen = np.concatenate([rng.choice(nb - 1, size=take - 1, replace=False),
                                     [nb - 1]]).astype(np.int32)
        prev = list(chosen)
        rng.shuffle(chosen)
        ids[r, :take] = chosen
    return ids, rl


def _host_tables(ids, rl, nn, kb, page_table, ps):
    """Ascending INT32_MAX-padded tables, physical blocks and live lengths by
    their definitions, from the host's own ids (rows with nb <= kb: every
    block)."""
    R = ids.shape[0]
    table = np.full((R, kb), IMAX, np.int32)
    phys = np.full((R, kb), IMAX, np.int32)
    vl = np.zeros(R, np.int32)
    for r in range(R):
        nb = int((rl[r] + 7) // 8)
        sel = list(range(nb)) if nb <= kb else sorted({int(x) for x in ids[r] if 0 <= x < nb})
        for i, blk in enumerate(sel):
            tok = blk * 8
            table[r, i] = blk
            phys[r, i] = (int(page_table[r // nn, tok // ps]) * ps + tok % ps) // 8
            vl[r] += min(8, int(rl[r]) - tok)
    return table, phys, vl


@pytest.mark.parametrize("ctx,kb,ps,nn", [
    ([20000, 3000, 9001], 512, 64, 2),
    ([20003, 700, 40000], 256, 128, 3),
    ([12000, 5001], 512, 64, 4),
    ([3000, 2100], 16, 64, 4),
    ([0, 2, 9, 5000], 16, 64, 4),     # empty request, rows with no or few keys
    ([3000, 20000], 64, 128, 1),      # every unit a lone row
])
def test_paired_sparse_pass(ctx, kb, ps, nn):
    """Row pairing: the paired sort gives the unpaired sort's tables bit for
    bit plus the oracle's union of each unit; the paired sparse logits equal
    the unpaired ones bitwise (FP32, FP16, BF16) and the oracle within the
    logits tolerance."""
    import dsa_sparse_attention_paged_gb300 as D
    B = len(ctx)
    R = B * nn
    case = make(B, nn, ctx, ps, "normal", seed=900 + kb + nn)
    d = to_dev(case)
    ws = D.Workspace(R)
    ids, rl = _verify_ids(ctx, nn, kb, seed=kb + nn)
    t_ref, p_ref, v_ref = _host_tables(ids, rl, nn, kb, case["page_table"], ps)
    u_ref = O.pair_union(t_ref, p_ref, nn)

    ids1 = torch.from_numpy(ids).cuda()
    ids2 = ids1.clone()
    phys1 = torch.empty((R, kb), dtype=torch.int32, device="cuda")
    vl1 = torch.empty((R,), dtype=torch.int32, device="cuda")
    D.sort_candidate_blocks(ids1, d["context_lens"], nn, d["page_table"], ps, ws,
                            phys_blocks=phys1, valid_lens=vl1)
    U = D.pair_units(B, nn)
    assert U == B * ((nn + 1) // 2)
    union = (torch.full((U, 2 * kb), 7, dtype=torch.int32, device="cuda"),
             torch.full((U, 2 * kb), 7, dtype=torch.int32, device="cuda"),
             torch.full((U,), 7, dtype=torch.int32, device="cuda"))
    phys2 = torch.empty((R, kb), dtype=torch.int32, device="cuda")
    vl2 = torch.empty((R,), dtype=torch.int32, device="cuda")
    D.sort_candidate_blocks_paired(ids2, d["context_lens"], nn, d["page_table"], ps, ws,
                                   valid_lens=vl2, union=union, phys_blocks=phys2)
    torch.cuda.synchronize()
    assert ws.status() == 0
    np.testing.assert_array_equal(ids1.cpu().numpy(), t_ref)
    np.testing.assert_array_equal(phys1.cpu().numpy(), p_ref)
    np.testing.assert_array_equal(vl1.cpu().numpy(), v_ref)
    assert torch.equal(ids2, ids1) and torch.equal(phys2, phys1) and torch.equal(vl2, vl1)
    for got, want in zip(union, u_ref):
        np.testing.assert_array_equal(got.cpu().numpy(), want)

    rtr = np.arange(R, dtype=np.int32) // nn
    ref_sp = O.sparse_logits(case["q"], case["kv"], case["kscale"], case["weights"],
                             case["page_table"], rl, rtr, ps, t_ref)
    masked = np.isneginf(ref_sp)
    for dt, view in ((D.OUT_F32, torch.int32), (D.OUT_F16, torch.int16),
                     (D.OUT_BF16, torch.int16)):
        stride = kb * 8 + 24
        tdt = {D.OUT_F32: torch.float32, D.OUT_F16: torch.float16,
               D.OUT_BF16: torch.bfloat16}[dt]
        o1 = torch.full((R, stride), 3.0, dtype=tdt, device="cuda")
        o2 = torch.full((R, stride), 3.0, dtype=tdt, device="cuda")
        D.sparse_mqa_logits(d["q"], d["kv"], d["kscale"], d["weights"], d["page_table"],
                            d["context_lens"], nn, ids1, ws, out=o1, out_dtype=dt,
                            phys_blocks=phys1, valid_lens=vl1)
        D.sparse_mqa_logits_paired(d["q"], d["kv"], d["kscale"], d["weights"],
                                   d["page_table"], d["context_lens"], nn, kb, union, vl2, ws,
                                   out=o2, out_dtype=dt)
        torch.cuda.synchronize()
        assert ws.status() == 0
        assert torch.equal(o2.view(view), o1.view(view)), dt
        # nothing written past kb*8
        assert (o2[:, kb * 8:].float() == 3.0).all()
        if dt == D.OUT_F32:
            S2 = o2[:, :kb * 8].cpu().numpy()
            np.testing.assert_array_equal(np.isneginf(S2), masked)
            assert_close(S2[~masked], ref_sp[~masked], "paired sparse logits")


@pytest.mark.parametrize("ps,nn", [(32, 2), (8, 3), (256, 1)])
def test_sort_tables_other_page_sizes(ps, nn):
    """The sorts' physical blocks for page sizes the sparse kernel does not
    take (its word-wise page loads cover power-of-two pages of 64 tokens and
    more; other sizes read the page table per block): unpaired and paired
    tables against their definitions and the oracle's union."""
    import dsa_sparse_attention_paged_gb300 as D
    ctx = [9000, 20001, 700]
    kb = 128
    B = len(ctx)
    R = B * nn
    case = make(B, nn, ctx, ps, "normal", seed=77 + ps)
    d = to_dev(case)
    ws = D.Workspace(R)
    ids, rl = _verify_ids(ctx, nn, kb, seed=ps)
    t_ref, p_ref, v_ref = _host_tables(ids, rl, nn, kb, case["page_table"], ps)
    ids1 = torch.from_numpy(ids).cuda()
    phys1 = torch.empty((R, kb), dtype=torch.int32, device="cuda")
    vl1 = torch.empty((R,), dtype=torch.int32, device="cuda")
    D.sort_candidate_blocks(ids1, d["context_lens"], nn, d["page_table"], ps, ws,
                            phys_blocks=phys1, valid_lens=vl1)
    U = D.pair_units(B, nn)
    union = tuple(torch.empty(sh, dtype=torch.int32, device="cuda")
                  for sh in ((U, 2 * kb), (U, 2 * kb), (U,)))
    ids2 = torch.from_numpy(ids).cuda()
    phys2 = torch.empty((R, kb), dtype=torch.int32, device="cuda")
    vl2 = torch.empty((R,), dtype=torch.int32, device="cuda")
    D.sort_candidate_blocks_paired(ids2, d["context_lens"], nn, d["page_table"], ps, ws,
                                   valid_lens=vl2, union=union, phys_blocks=phys2)
    torch.cuda.synchronize()
    assert ws.status() == 0
    for t, ph, v in ((ids1, phys1, vl1), (ids2, phys2, vl2)):
        np.testing.assert_array_equal(t.cpu().numpy(), t_ref)
        np.testing.assert_array_equal(ph.cpu().numpy(), p_ref)
        np.testing.assert_array_equal(v.cpu().numpy(), v_ref)
    for got, want in zip(union, O.pair_union(t_ref, p_ref, nn)):
        np.testing.assert_array_equal(got.cpu().numpy(), want)
