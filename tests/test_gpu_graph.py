"""The decode step captured once in a CUDA graph and replayed after context
lengths, queries and head weights were rewritten in place: the same results
as an eager step on those values, and the oracle's top-2048 of the scores."""
import numpy as np
import pytest
import torch

import synthetic as S
from oracle import oracle as O
from tests.helpers import sets_equal, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("pair_rows", [False, True])
def test_graph_replay_follows_inputs_rewritten_in_place(pair_rows):
    from dsa_sparse_attention_paged_gb300.pipeline import DecodePlan
    # pages for 20000 keys in every request; each replay picks its own lengths
    a = S.generate(S.Workload("graph a", 3, 2, [20000] * 3, 64, "mixed", 91))
    b = S.generate(S.Workload("graph b", 3, 2, [20000] * 3, 64, "normal", 92))
    d = to_dev(a)
    d["context_lens"].copy_(torch.tensor([20000, 9000, 3000], dtype=torch.int32))
    plan = DecodePlan(3, 2, 20000, 64, k=2048, kb=256, pair_rows=pair_rows)
    plan.capture(d["q"], d["kv"], d["kscale"], d["weights"], d["page_table"], d["context_lens"])

    def replay_and_compare():
        g_dense, g_sparse = plan.replay()
        torch.cuda.synchronize()
        assert plan.ws.status() == 0
        gd, gs = g_dense.cpu().numpy().copy(), g_sparse.cpu().numpy().copy()
        rl = O.row_lens(d["context_lens"].cpu().numpy(), 2)
        L = plan.logits.cpu().numpy()
        live = np.arange(plan.stride)[None, :] < rl[:, None]
        assert sets_equal(gd, O.topk(np.where(live, L, np.nan).astype(np.float32), rl, 2048))
        e_dense, e_sparse = plan.step(d["q"], d["kv"], d["kscale"], d["weights"],
                                      d["page_table"], d["context_lens"])
        torch.cuda.synchronize()
        assert sets_equal(gd, e_dense.cpu().numpy())
        assert sets_equal(gs, e_sparse.cpu().numpy())

    replay_and_compare()
    d["context_lens"].copy_(torch.tensor([7000, 20000, 100], dtype=torch.int32))
    d["q"].copy_(torch.from_numpy(b["q"]))
    d["weights"].copy_(torch.from_numpy(b["weights"]))
    replay_and_compare()


def test_host_pipeline_matches_eager_steps():
    """Host-to-host steps two in flight (two slots, each a captured graph of
    copies + kernels + copies): every step's host outputs equal an eager step
    on the same inputs.  Each slot keeps its pinned buffers; their contents
    change between steps (lengths, queries, weights), so the later steps are
    graph replays over rewritten host memory."""
    from dsa_sparse_attention_paged_gb300.pipeline import DecodePlan, HostStepPipeline
    cases = [S.generate(S.Workload("pipe %d" % i, 3, 2, [20000] * 3, 64, dist, 300 + i))
             for i, dist in enumerate(("mixed", "normal", "mixed"))]
    lens = ([20000, 9000, 3000], [7000, 20000, 100], [15000, 15000, 15000])
    d = to_dev(cases[0])  # the K cache is the first case's; pages cover 20000 keys
    pipe = HostStepPipeline(3, 2, 20000, 64, d["kv"], d["kscale"], k=2048, kb=256)
    c0 = cases[0]
    slots = [({"q": torch.empty(c0["q"].shape, dtype=torch.uint8).pin_memory(),
               "weights": torch.empty(c0["weights"].shape, dtype=torch.float32).pin_memory(),
               "context_lens": torch.empty((3,), dtype=torch.int32).pin_memory(),
               "page_table": torch.from_numpy(c0["page_table"]).pin_memory()},
              (torch.empty((6, 2048), dtype=torch.int32).pin_memory(),
               torch.empty((6, 2048), dtype=torch.int32).pin_memory())) for _ in range(2)]
    plan = DecodePlan(3, 2, 20000, 64, k=2048, kb=256)

    def expect(j):
        c = cases[j]
        dense, sparse = plan.step(torch.from_numpy(c["q"]).cuda(), d["kv"], d["kscale"],
                                  torch.from_numpy(c["weights"]).cuda(), d["page_table"],
                                  torch.tensor(lens[j], dtype=torch.int32, device="cuda"))
        torch.cuda.synchronize()
        return dense.cpu().numpy(), sparse.cpu().numpy()

    order = [0, 1, 2, 1, 0, 2, 2, 0]
    for i, j in enumerate(order):
        hin, hout = slots[i % 2]
        if i >= 2:  # the slot's previous step: outputs final, inputs free
            pipe.wait(i - 2)
            e_dense, e_sparse = expect(order[i - 2])
            assert sets_equal(hout[0].numpy(), e_dense)
            assert sets_equal(hout[1].numpy(), e_sparse)
        hin["q"].copy_(torch.from_numpy(cases[j]["q"]))
        hin["weights"].copy_(torch.from_numpy(cases[j]["weights"]))
        hin["context_lens"].copy_(torch.tensor(lens[j], dtype=torch.int32))
        pipe.submit(hin["q"], hin["weights"], hin["context_lens"], hin["page_table"], *hout)
    pipe.synchronize()
    for p in pipe.plans:
        assert p.ws.status() == 0
    for i in (len(order) - 2, len(order) - 1):
        e_dense, e_sparse = expect(order[i])
        hout = slots[i % 2][1]
        assert sets_equal(hout[0].numpy(), e_dense)
        assert sets_equal(hout[1].numpy(), e_sparse)


@pytest.mark.parametrize("B,nn,L,ps,kb", [(4, 1, 40000, 64, 512), (3, 2, 20001, 128, 256)])
def test_one_call_step_equals_separate_calls(B, nn, L, ps, kb):
    """``dsa_decode_step`` (one library call for the whole step) writes what
    the four separate calls write: bit for bit the logits, the cleared
    histogram, the sorted table, physical blocks, live lengths and the FP16
    sparse scores, and the same two index sets (in any order); a second step
    on lengths rewritten in place reuses the argument block and follows them."""
    from dsa_sparse_attention_paged_gb300.pipeline import DecodePlan
    case = S.generate(S.Workload("one call", B, nn, [L] * B, ps, "mixed", 777 + B))
    d = to_dev(case)
    lens2 = torch.tensor([max(1, L - 997 * (i + 1)) for i in range(B)], dtype=torch.int32,
                         device="cuda")
    plans = [DecodePlan(B, nn, L, ps, k=2048, kb=kb) for _ in range(2)]
    assert plans[0].fused_table
    ctx = d["context_lens"].clone()
    for it in range(2):
        if it == 1:
            ctx.copy_(lens2)  # rewritten in place: the same argument block
        inp = (d["q"], d["kv"], d["kscale"], d["weights"], d["page_table"], ctx)
        outs = []
        for i, plan in enumerate(plans):
            plan.logits.fill_(float("nan"))
            plan.step(*inp, events=None if i == 0 else {})  # events: the separate calls
            torch.cuda.synchronize()
            assert plan.ws.status() == 0
            outs.append([t.cpu() for t in (plan.logits, plan.hist, plan.topk_idx, plan.block_ids,
                                           plan.phys, plan.valid_lens, plan.sparse,
                                           plan.sparse_idx)])
        bits = {torch.float32: torch.int32, torch.float16: torch.int16}
        for i, (a, b) in enumerate(zip(*outs)):
            if i in (2, 7):  # index sets: their order is unspecified
                assert sets_equal(a.numpy(), b.numpy())
            else:
                assert torch.equal(a.view(bits.get(a.dtype, a.dtype)),
                                   b.view(bits.get(b.dtype, b.dtype)))
        rl = O.row_lens(ctx.cpu().numpy(), nn)
        L_np = outs[0][0].numpy()
        assert sets_equal(outs[0][2].numpy(), O.topk(L_np, rl, 2048))
