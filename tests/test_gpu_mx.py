"""MXFP4 index keys (block-scaled E2M1 codes + UE8M0 exponents) through the
block-scaled tensor-core path, against the oracle's MXFP4 logits.

Sources: SGLang PR #38944 (Hopper prefill commit text: block-scaled E2M1
index keys), vLLM PR #52696 ("Why"; the MXFP4 indexer-cache layout)."""
import numpy as np
import pytest
import torch

import synthetic as S
from oracle import oracle as O
from tests.helpers import assert_close, live_mask, to_dev

pytestmark = pytest.mark.gpu

# E2M1 codes whose values are multiples of 0.5 up to 2 (0, 0.5, 1, 1.5, 2 and
# their negatives) and block exponents 2^-1 .. 2^1
_SMALL_CODES = np.array([0, 1, 2, 3, 4, 9, 10, 11, 12], np.uint8)


def _mx_case(B, nn, ctx, ps, dist, seed):
    return S.generate(S.Workload("mx", B, nn, list(ctx), ps, dist, seed, key_format="mxfp4"))


def _run_mx(D, d, nn, stride, hist=None):
    ws = D.Workspace(d["q"].shape[0])
    R = d["q"].shape[0]
    logits = torch.full((R, stride), float("nan"), dtype=torch.float32, device="cuda")
    D.paged_mqa_logits_mx(d["q"], d["k_codes"], d["k_exp"], d["weights"], d["page_table"],
                          d["context_lens"], nn, ws, logits=logits, histogram=hist)
    torch.cuda.synchronize()
    assert ws.status() == 0
    return logits.cpu().numpy()


@pytest.mark.parametrize("B,nn,ctx,ps,dist", [
    (1, 1, [5000], 64, "normal"),
    (3, 1, [3000, 129, 7000], 128, "mixed"),
    (3, 2, [4100, 1, 2000], 64, "normal"),
    (2, 3, [9000, 300], 128, "normal"),
    (2, 4, [6000, 257], 64, "mixed"),
])
def test_mx_logits_match_oracle(B, nn, ctx, ps, dist):
    import dsa_sparse_attention_paged_gb300 as D
    c = _mx_case(B, nn, ctx, ps, dist, seed=500 + 7 * nn + B)
    d = to_dev(c)
    stride = (max(ctx) + 15) // 8 * 8
    L = _run_mx(D, d, nn, stride)
    ref = O.paged_mqa_logits_mx(c["q"], c["k_codes"], c["k_exp"], c["weights"], c["page_table"],
                                c["context_lens"], nn, ps, logits_stride=stride)
    live, rl = live_mask(c["context_lens"], nn, stride)
    assert_close(L[live], ref[live], "MXFP4 logits")
    assert np.isnan(L[~live]).all(), "dead columns were written"


def test_mx_histogram_bitwise_and_logits_unchanged():
    import dsa_sparse_attention_paged_gb300 as D
    c = _mx_case(2, 2, [20000, 7000], 64, "mixed", seed=77)
    d = to_dev(c)
    stride = 20008
    L0 = _run_mx(D, d, 2, stride)
    hist = torch.zeros((4, 1024), dtype=torch.int32, device="cuda")
    L1 = _run_mx(D, d, 2, stride, hist)
    live, rl = live_mask(c["context_lens"], 2, stride)
    np.testing.assert_array_equal(L0[live].view(np.uint32), L1[live].view(np.uint32))
    want = O.histogram(np.where(live, L1, np.nan).astype(np.float32), rl)
    np.testing.assert_array_equal(hist.cpu().numpy(), want)
    _run_mx(D, d, 2, stride, hist)  # accumulates
    np.testing.assert_array_equal(hist.cpu().numpy(), 2 * want)


def _intexact_mx(B, nn, ctx, ps, seed, equal_exponents=False):
    """Integer-exact MXFP4 inputs: q in {-2..2}, key values multiples of 0.25
    up to 4, head weights in {+-1/2, +-1, +-2}: every product and partial sum
    is exact in FP32, so any summation order gives the same float."""
    c = S.generate(S.Workload("mx exact", B, nn, list(ctx), ps, "intexact", seed,
                              key_format="mxfp4"))
    rng = np.random.default_rng(seed)
    P = c["num_pages"]
    nib = _SMALL_CODES[rng.integers(0, len(_SMALL_CODES), (P, ps, 128))]
    c["k_codes"] = np.ascontiguousarray((nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8))
    if equal_exponents:
        e = rng.integers(126, 129, (P, ps, 1)).astype(np.uint8)
        c["k_exp"] = np.ascontiguousarray(np.repeat(e, 4, axis=2))
    else:
        c["k_exp"] = rng.integers(126, 129, (P, ps, 4)).astype(np.uint8)
    return c, nib


@pytest.mark.parametrize("nn", [1, 2, 4])
def test_mx_integer_exact_bitwise(nn):
    import dsa_sparse_attention_paged_gb300 as D
    c, _ = _intexact_mx(2, nn, [3000, 700], 64, seed=91 + nn)
    d = to_dev(c)
    stride = 3008
    L = _run_mx(D, d, nn, stride)
    ref = O.paged_mqa_logits_mx(c["q"], c["k_codes"], c["k_exp"], c["weights"], c["page_table"],
                                c["context_lens"], nn, 64, logits_stride=stride)
    live, _ = live_mask(c["context_lens"], nn, stride)
    np.testing.assert_array_equal(L[live].view(np.uint32), ref[live].view(np.uint32))


def test_mx_one_hot_queries_pick_one_code_and_its_block_exponent():
    """q one-hot at (head h, dimension d) with weight 1 on head h: the logit of
    token t is ReLU(E2M1(code[t][d]) * 2^(e[t][d / 32] - 127)) -- nibble order
    and block index against the oracle."""
    import dsa_sparse_attention_paged_gb300 as D
    c, _ = _intexact_mx(1, 1, [2048], 128, seed=5)
    q = np.zeros_like(c["q"])
    w = np.zeros_like(c["weights"])
    for trial, (h, dd) in enumerate([(0, 0), (3, 1), (31, 33), (7, 64), (12, 127), (20, 96)]):
        q[:] = 0
        q[0, h, dd] = 0x38  # E4M3 1.0
        w[:] = 0
        w[0, h] = 1.0
        c2 = dict(c, q=q.copy(), weights=w.copy())
        L = _run_mx(D, to_dev(c2), 1, 2048)
        ref = O.paged_mqa_logits_mx(c2["q"], c2["k_codes"], c2["k_exp"], c2["weights"],
                                    c2["page_table"], c2["context_lens"], 1, 128,
                                    logits_stride=2048)
        np.testing.assert_array_equal(L.view(np.uint32), ref.view(np.uint32), str((h, dd)))
        assert (ref > 0).any() and (ref == 0).any(), "a useful one-hot case"


def test_mx_equals_fp8_path_when_block_exponents_agree():
    """With one exponent e for all four blocks of a token, the MXFP4 key is the
    FP8 key with the same code values and kscale 2^(e - 127): both library
    paths give bitwise equal logits on integer-exact inputs."""
    import dsa_sparse_attention_paged_gb300 as D
    c, nib = _intexact_mx(2, 2, [4000, 900], 64, seed=17, equal_exponents=True)
    vals = np.array([O.e2m1(int(x)) for x in range(16)], np.float32)[nib]
    kv = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    kscale = np.ldexp(1.0, c["k_exp"][..., 0].astype(np.int32) - 127).astype(np.float32)
    d = to_dev(dict(c, kv=np.ascontiguousarray(kv), kscale=np.ascontiguousarray(kscale)))
    stride = 4008
    Lmx = _run_mx(D, d, 2, stride)
    ws = D.Workspace(4)
    L8 = torch.full((4, stride), float("nan"), dtype=torch.float32, device="cuda")
    D.paged_mqa_logits(d["q"], d["kv"], d["kscale"], d["weights"], d["page_table"],
                       d["context_lens"], 2, ws, logits=L8)
    torch.cuda.synchronize()
    live, _ = live_mask(c["context_lens"], 2, stride)
    np.testing.assert_array_equal(Lmx[live].view(np.uint32), L8.cpu().numpy()[live].view(np.uint32))


def test_mx_rejects_bad_arguments():
    import ctypes
    import dsa_sparse_attention_paged_gb300 as D
    c = _mx_case(1, 1, [256], 64, "normal", seed=3)
    d = to_dev(c)
    ws = D.Workspace(1)
    L = torch.empty((1, 256), dtype=torch.float32, device="cuda")
    codes_off = torch.empty(d["k_codes"].numel() + 16, dtype=torch.uint8, device="cuda")[16:]
    args = lambda codes, nn=1, H=32: (  # noqa: E731
        ctypes.c_void_p(d["q"].data_ptr()), ctypes.c_void_p(codes), ctypes.c_void_p(d["k_exp"].data_ptr()),
        ctypes.c_void_p(d["weights"].data_ptr()), ctypes.c_void_p(d["page_table"].data_ptr()),
        d["page_table"].stride(0), ctypes.c_void_p(d["context_lens"].data_ptr()), 1, nn, H, 128, 64,
        c["num_pages"], ctypes.c_void_p(L.data_ptr()), 256, None, ws.ptr, ws.nbytes, None)
    assert D.lib.dsa_paged_mqa_logits_mx(*args(codes_off.data_ptr())) == 3  # 16 B: misaligned
    assert D.lib.dsa_paged_mqa_logits_mx(*args(d["k_codes"].data_ptr(), nn=5)) == 2
    assert D.lib.dsa_paged_mqa_logits_mx(*args(d["k_codes"].data_ptr(), H=16)) == 2
    assert D.lib.dsa_paged_mqa_logits_mx(*args(None)) == 1
