"""Full-size parity on the five named workloads, in the launch configuration
the bench times (DecodePlan): every live logit against the oracle (one
request per task of a process pool); histograms, top-k sets, block tables
and the FP16 select exactly, on the GPU's own logits; sparse logits bitwise
against the dense logits at the chosen positions.  MXFP4 keys at the
largest workload's shape: sampled logits against the oracle one by one."""
import multiprocessing as mp
import os

import numpy as np
import pytest
import torch

import synthetic as S
from oracle import oracle as O
from tests.helpers import assert_close, sets_equal, to_dev

pytestmark = pytest.mark.gpu

_CASE_KEYS = ("q", "kv", "kscale", "weights", "page_table", "context_lens")


def _oracle_request_logits(args):
    """One request's dense logits [next_n][stride] from the case saved in
    `folder` (memory-mapped, so the workers share one copy)."""
    folder, b, nn, ps, stride = args
    c = {k: np.load(os.path.join(folder, k + ".npy"), mmap_mode="r") for k in _CASE_KEYS}
    return b, O.paged_mqa_logits(c["q"][b * nn:(b + 1) * nn], c["kv"], c["kscale"],
                                 c["weights"][b * nn:(b + 1) * nn], c["page_table"][b:b + 1],
                                 c["context_lens"][b:b + 1], nn, ps, logits_stride=stride)


@pytest.fixture(scope="module")
def oracle_pool():
    ctx = mp.get_context("spawn")  # no fork after the GPU is in use
    with ctx.Pool(min(16, os.cpu_count() or 1)) as pool:
        yield pool


def _oracle_logits_all(case, nn, ps, stride, folder, pool):
    for k in _CASE_KEYS:
        np.save(os.path.join(folder, k + ".npy"), np.ascontiguousarray(case[k]))
    B = len(case["context_lens"])
    ref = np.full((B * nn, stride), np.nan, np.float32)
    for b, Lb in pool.imap_unordered(_oracle_request_logits,
                                      [(folder, b, nn, ps, stride) for b in range(B)]):
        ref[b * nn:(b + 1) * nn] = Lb
    return ref


@pytest.mark.parametrize("name", ["c0", "c1", "c2", "c3", "c3u", "c4"])
def test_full_size_workload(name, oracle_pool, tmp_path):
    from dsa_sparse_attention_paged_gb300.pipeline import DecodePlan
    w = S.named(name)
    case = S.generate(w)
    d = to_dev(case)
    nn, ps = w.next_n, w.page_size
    plan = DecodePlan(w.B, nn, max(w.context_lens), ps, k=2048, kb=512, two_level=True,
                      pair_rows=nn > 1)
    dense_idx, sparse_idx = plan.step(d["q"], d["kv"], d["kscale"], d["weights"],
                                      d["page_table"], d["context_lens"])
    torch.cuda.synchronize()
    assert plan.ws.status() == 0
    R = w.R
    rl = O.row_lens(case["context_lens"], nn)
    L = plan.logits.cpu().numpy()

    # logits: every live position against the oracle
    ref = _oracle_logits_all(case, nn, ps, plan.stride, str(tmp_path), oracle_pool)
    live = np.arange(plan.stride)[None, :] < rl[:, None]
    assert_close(L[live], ref[live], f"{name} logits")

    # histogram of the GPU's own logits (the plan's top-k reset it, so rerun)
    hist = torch.zeros((R, 1024), dtype=torch.int32, device="cuda")
    import dsa_sparse_attention_paged_gb300 as D
    L2 = D.paged_mqa_logits(d["q"], d["kv"], d["kscale"], d["weights"], d["page_table"],
                            d["context_lens"], nn, plan.ws, logits_stride=plan.stride,
                            histogram=hist)
    torch.cuda.synchronize()
    live = np.arange(plan.stride)[None, :] < rl[:, None]
    Lm = np.where(live, L, np.nan).astype(np.float32)
    np.testing.assert_array_equal(L2.cpu().numpy()[live], L[live])
    np.testing.assert_array_equal(hist.cpu().numpy(), O.histogram(Lm, rl))
    if name == "c2":  # 'mixed' spans fine, unit and saturating bins
        h = hist.cpu().numpy().sum(0)
        assert h[0] + h[1023] > 0 and h[1:207].sum() + h[817:1023].sum() > 0
        assert h[208:816].sum() > 0

    # dense top-2048
    assert sets_equal(dense_idx.cpu().numpy(), O.topk(Lm, rl, 2048))

    # two-level chain: block maxima of the GPU's own logits (selected inside
    # the select when rows fit a cluster, else written by the logits pass)
    kb = plan.kb
    nb = (rl + 7) // 8
    A = O.block_amax8(Lm, rl, skip_le=kb, amax_stride=plan.amax_stride, fill=0.0)
    if plan.amax is not None:
        Ag = plan.amax.cpu().numpy()
        for r in range(R):
            if nb[r] > kb:
                np.testing.assert_array_equal(Ag[r, :nb[r]], A[r, :nb[r]])
    rtr = np.arange(R, dtype=np.int32) // nn
    t_ref, p_ref, v_ref = O.block_table(A, rl, rtr, kb, case["page_table"], ps)
    np.testing.assert_array_equal(plan.block_ids.cpu().numpy(), t_ref)
    np.testing.assert_array_equal(plan.phys.cpu().numpy(), p_ref)
    np.testing.assert_array_equal(plan.valid_lens.cpu().numpy(), v_ref)
    if plan.union is not None:  # next_n > 1: two rows of a request per K pass
        for got, want in zip(plan.union, O.pair_union(t_ref, p_ref, nn)):
            np.testing.assert_array_equal(got.cpu().numpy(), want)
    SP16 = plan.sparse.cpu().numpy().view(np.uint16)
    pos = np.arange(kb * 8)
    for r in range(R):
        tok = t_ref[r, pos // 8].astype(np.int64) * 8 + pos % 8
        n_live = v_ref[r]
        np.testing.assert_array_equal(SP16[r, :n_live], O.fp16_rn_array(L[r, tok[:n_live]]))
        assert (SP16[r, n_live:] == 0xFC00).all()
    assert sets_equal(sparse_idx.cpu().numpy(), O.topk_fp16(SP16, v_ref, 2048, t_ref))


def test_full_size_mxfp4_keys_largest_shape():
    """MXFP4 keys at B=32, L=131072 (page 64): the launch the bench times for
    the MXFP4 key stream; 8192 sampled live logits plus every row's first and
    last column against the oracle, and the fused histogram on the GPU's own
    logits."""
    import dsa_sparse_attention_paged_gb300 as D
    w = S.named("c2")
    case = S.generate(w)
    g = torch.Generator().manual_seed(w.seed + 1000)
    P = case["num_pages"]
    codes = torch.randint(0, 256, (P, w.page_size, 64), generator=g, dtype=torch.uint8)
    exps = torch.randint(125, 130, (P, w.page_size, 4), generator=g, dtype=torch.uint8)
    d = to_dev(case)
    R, stride = w.R, 131072
    ws = D.Workspace(R)
    hist = torch.zeros((R, 1024), dtype=torch.int32, device="cuda")
    L = D.paged_mqa_logits_mx(d["q"], codes.cuda(), exps.cuda(), d["weights"], d["page_table"],
                              d["context_lens"], 1, ws, logits_stride=stride, histogram=hist)
    torch.cuda.synchronize()
    assert ws.status() == 0
    L = L.cpu().numpy()
    rl = O.row_lens(case["context_lens"], 1)
    rng = np.random.default_rng(2)
    rows = rng.integers(0, R, 8192)
    cols = (rng.random(8192) * rl[rows]).astype(np.int64)
    rows = np.concatenate([rows, np.arange(R), np.arange(R)])
    cols = np.concatenate([cols, np.zeros(R, np.int64), rl - 1])
    ref = O.logits_at_mx(case["q"], codes.numpy(), exps.numpy(), case["weights"],
                         case["page_table"], 1, w.page_size, rows, cols)
    assert_close(L[rows, cols], ref, "MXFP4 logits")
    np.testing.assert_array_equal(hist.cpu().numpy(), O.histogram(L, rl))
