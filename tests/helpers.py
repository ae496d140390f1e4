"""Shared test helpers: move a synthetic case to the GPU and run the oracle."""
import numpy as np
import torch

import synthetic as S
from oracle import oracle as O

TOL_ABS = 1e-3
TOL_REL = 1e-3


def to_dev(case, device="cuda"):
    d = {}
    for k, v in case.items():
        if isinstance(v, np.ndarray):
            d[k] = torch.from_numpy(np.ascontiguousarray(v)).to(device)
        else:
            d[k] = v
    return d


def assert_close(gpu, ref, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(gpu - ref)
    bound = TOL_ABS + TOL_REL * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} mismatches, first at {tuple(i)}: "
                             f"gpu={gpu[tuple(i)]} ref={ref[tuple(i)]}")


def live_mask(ctx, next_n, stride):
    rl = O.row_lens(ctx, next_n)
    return np.arange(stride)[None, :] < rl[:, None], rl


def sets_equal(a, b):
    """Row-wise set equality of index arrays (order-free, -1 padding kept)."""
    a = np.sort(np.asarray(a), axis=1)
    b = np.sort(np.asarray(b), axis=1)
    return np.array_equal(a, b)


def make(B, next_n, ctx, ps, dist="normal", seed=1):
    return S.generate(S.Workload("test", B, next_n, list(ctx), ps, dist, seed))
