"""One indexer decode step as a fixed sequence of C-ABI calls.

``DecodePlan`` plays the role of SGLang's ``FusedDecodePlan`` (DeepGEMM PR #94,
cross-referenced SGLang commit 7e252c5): it is built once per shape, owns the
step's device buffers and the workspace, and each ``step`` runs

  source layer   paged MQA logits + fused coarse histogram          (1 launch)
                 histogram-driven exact top-k of the logits rows
                 (resets the hist) and, in the same launch, top-kb
                 of their block maxima over 8 scores (amax8 +
                 top-kb fused into the select)                     (1 launch
                 for rows up to 131072 scores; longer rows: block
                 maxima fused into the logits pass and a second
                 problem of the batched select instead)
  level one      sort_candidate_blocks -> table, phys, valid lens   (inside the
                 select launch for rows a cluster takes; else 1 launch;
                 pair_rows: the paired sort, which also emits the
                 union of each two-row unit's tables)
  consumer       sparse MQA logits over the table, FP16 output      (1 launch)
                 (pair_rows: two rows of a request per K pass)
                 FP16 top-k with the fused table transform          (1 launch)

following SGLang PR #38944 ("What this enables": the source layer publishes an
ascending block table; the consumer scores only those blocks and selects
inside that row).  Everything runs in the library's kernels on one stream.
"""
from __future__ import annotations

import torch

from . import (OUT_F16, Workspace, coarse_hist_topk, coarse_hist_topk_batch,
               coarse_hist_topk_batch_launches, coarse_hist_topk_launches, paged_mqa_logits,
               pair_units, sort_candidate_blocks, sort_candidate_blocks_paired,
               sparse_mqa_logits, sparse_mqa_logits_paired, topk_fp16)


class DecodePlan:

    def __init__(self, B, next_n, max_context, page_size, k=2048, kb=512, two_level=True,
                 pair_rows=False, device="cuda"):
        """``pair_rows`` scores two rows of a request per K pass in the sparse
        step (same results, bitwise).  It pays when the two rows' tables share
        most blocks (draft rows of one request); on independent rows the union
        is twice a table and the unpaired pass is faster."""
        self.B, self.next_n, self.page_size = B, next_n, page_size
        self.pair_rows = bool(pair_rows) and next_n > 1
        self.R = B * next_n
        self.k, self.kb, self.two_level = k, kb, two_level
        # row stride padded to 8 floats: 32-byte aligned rows for the vector loads
        self.stride = (int(max_context) + 7) // 8 * 8
        dev = torch.device(device)
        R = self.R
        # block maxima selected inside the logits-row select (rows a cluster
        # takes), else written by the logits pass and selected as a second problem
        self.fused_blocks = two_level and coarse_hist_topk_batch_launches(
            [(self.stride, True, R)]) == 1
        self.ws = Workspace(2 * R if two_level and not self.fused_blocks else R, device=dev)
        self.logits = torch.empty((R, self.stride), dtype=torch.float32, device=dev)
        self.hist = torch.zeros((R, 1024), dtype=torch.int32, device=dev)
        self.topk_idx = torch.empty((R, k), dtype=torch.int32, device=dev)
        self.amax = None
        if two_level:
            self.amax_stride = (self.stride + 7) // 8
            self.amax = (None if self.fused_blocks else
                         torch.empty((R, self.amax_stride), dtype=torch.float32, device=dev))
            self.block_ids = torch.empty((R, kb), dtype=torch.int32, device=dev)
            self.phys = torch.empty((R, kb), dtype=torch.int32, device=dev)
            self.valid_lens = torch.empty((R,), dtype=torch.int32, device=dev)
            self.sparse = torch.empty((R, kb * 8), dtype=torch.float16, device=dev)
            self.sparse_idx = torch.empty((R, k), dtype=torch.int32, device=dev)
            self.union = None
            if self.pair_rows:
                U = pair_units(B, next_n)
                self.union = (torch.empty((U, 2 * kb), dtype=torch.int32, device=dev),
                              torch.empty((U, 2 * kb), dtype=torch.int32, device=dev),
                              torch.empty((U,), dtype=torch.int32, device=dev))

    @property
    def launches_per_step(self) -> int:
        """Kernels of this library launched by one step."""
        if not self.two_level:
            return 1 + coarse_hist_topk_launches(self.stride, True)
        if self.fused_blocks:
            sel = coarse_hist_topk_batch_launches([(self.stride, True, self.R)])
        else:
            sel = coarse_hist_topk_batch_launches([(self.stride, True, self.R),
                                                   (self.amax_stride, False, self.R)])
        sort = 0 if self.fused_table else 1
        return 1 + sel + sort + 1 + 1

    @property
    def fused_table(self) -> bool:
        """The sorted block table comes out of the select launch (rows a
        cluster takes, unpaired rows): no separate sort launch."""
        return self.two_level and self.fused_blocks and self.union is None

    def step(self, q, kv, kscale, weights, page_table, context_lens, events=None):
        """Run one decode step.  ``events`` (optional dict name -> (start, end)
        CUDA events) brackets individual launches for per-kernel timing."""
        nn, ws = self.next_n, self.ws

        def mark(name, i):
            if events is not None and name in events:
                events[name][i].record()

        mark("logits", 0)
        paged_mqa_logits(q, kv, kscale, weights, page_table, context_lens, nn, ws,
                         logits=self.logits, histogram=self.hist, amax=self.amax,
                         amax_skip_if_blocks_le=self.kb)
        mark("logits", 1)
        if not self.two_level:
            mark("select", 0)
            coarse_hist_topk(self.logits, context_lens, nn, self.k, ws, histogram=self.hist,
                             reset_histogram=True, out=self.topk_idx)
            mark("select", 1)
            return self.topk_idx, None
        mark("select", 0)
        dense = dict(logits=self.logits, context_lens=context_lens, next_n=nn, k=self.k,
                     histogram=self.hist, reset_histogram=True, out=self.topk_idx)
        if self.fused_table:
            coarse_hist_topk_batch([dict(dense, block_k=self.kb, block_out=self.block_ids,
                                         block_page_table=page_table,
                                         block_page_size=self.page_size, block_phys=self.phys,
                                         block_valid_lens=self.valid_lens)], ws)
        elif self.fused_blocks:
            coarse_hist_topk_batch([dict(dense, block_k=self.kb, block_out=self.block_ids)], ws)
        else:
            coarse_hist_topk_batch([dense, dict(
                logits=self.amax, context_lens=context_lens, next_n=nn, k=self.kb, len_div=8,
                out=self.block_ids)], ws)
        mark("select", 1)
        mark("publish", 0)
        if self.fused_table:
            pass  # the select launch wrote the sorted table, physical blocks, live lengths
        elif self.union is not None:
            sort_candidate_blocks_paired(self.block_ids, context_lens, nn, page_table,
                                         self.page_size, ws, self.valid_lens, self.union,
                                         phys_blocks=self.phys)
        else:
            sort_candidate_blocks(self.block_ids, context_lens, nn, page_table, self.page_size,
                                  ws, phys_blocks=self.phys, valid_lens=self.valid_lens)
        mark("publish", 1)
        mark("consume", 0)
        if self.union is not None:
            sparse_mqa_logits_paired(q, kv, kscale, weights, page_table, context_lens, nn,
                                     self.kb, self.union, self.valid_lens, ws, out=self.sparse,
                                     out_dtype=OUT_F16)
        else:
            sparse_mqa_logits(q, kv, kscale, weights, page_table, context_lens, nn,
                              self.block_ids, ws, out=self.sparse, out_dtype=OUT_F16,
                              phys_blocks=self.phys, valid_lens=self.valid_lens)
        topk_fp16(self.sparse, self.valid_lens, self.k, ws, block_table=self.block_ids,
                  out=self.sparse_idx)
        mark("consume", 1)
        return self.topk_idx, self.sparse_idx

    def capture(self, q, kv, kscale, weights, page_table, context_lens, stream=None):
        """Capture one step into a CUDA graph (after one eager step that sets
        the kernels' launch attributes).  Every grid depends only on the plan's
        shape (B, next_n, the maximum stride, kb), and every kernel reads the
        context lengths from device memory, so the graph stays valid when the
        caller rewrites ``context_lens`` (within the maximum), ``q``,
        ``weights``, ``page_table`` or the cache contents in place: ``replay()``
        then runs the step on the new values.  Returns the graph."""
        self.step(q, kv, kscale, weights, page_table, context_lens)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            out = self.step(q, kv, kscale, weights, page_table, context_lens)
        self.graph = g
        self.graph_out = out
        return g

    def replay(self):
        """Run the captured step (see ``capture``); returns its outputs."""
        self.graph.replay()
        return self.graph_out


class HostStepPipeline:
    """Decode steps fed from and returned to host memory, with the copies of
    one step overlapped with the kernels of its neighbours.

    Two ``DecodePlan``s and two device copies of the per-step inputs (q,
    weights, context lengths, page table) alternate between steps.  ``submit``
    queues three things on three streams:

      input stream    host-to-device copy of the step's inputs into the idle
                      set, once the step that last read that set has finished
      compute stream  the step (``DecodePlan.step``), once its inputs are in
                      and the step that last wrote its plan's outputs has had
                      them copied out
      output stream   device-to-host copy of both index sets, once the step
                      has finished

    so step i+1's inputs travel while step i computes, and step i's results
    travel while step i+1 computes.  The K cache (``kv``, ``kscale``) is
    resident device state that both plans read.  Host tensors must be pinned
    and stay untouched until the step's ``wait``; the kernels and the results
    are those of ``DecodePlan.step``."""

    def __init__(self, B, next_n, max_context, page_size, kv, kscale, k=2048, kb=512,
                 device="cuda"):
        dev = torch.device(device)
        self.plans = [DecodePlan(B, next_n, max_context, page_size, k=k, kb=kb, two_level=True,
                                 device=dev) for _ in range(2)]
        self.kv, self.kscale = kv, kscale
        self.inputs = [None, None]
        self.s_in = torch.cuda.Stream(device=dev)
        self.s_compute = torch.cuda.Stream(device=dev)
        self.s_out = torch.cuda.Stream(device=dev)
        self.step_done = [None, None]   # per set: the last step that used it finished
        self.out_done = [None, None]    # per set: that step's outputs reached the host
        self.pending = {}               # step index -> out_done event
        self.n = 0
        # the plans' buffers were zeroed on the caller's stream
        ready = torch.cuda.Event()
        ready.record(torch.cuda.current_stream(dev))
        self.start_after(ready)

    @property
    def launches_per_step(self) -> int:
        return self.plans[0].launches_per_step

    def start_after(self, event):
        """Make every later submit wait for ``event`` (e.g. a timing mark)."""
        for st in (self.s_in, self.s_compute, self.s_out):
            st.wait_event(event)

    def record_all(self):
        """An event on each stream, after everything submitted so far."""
        evs = []
        for st in (self.s_in, self.s_compute, self.s_out):
            e = torch.cuda.Event()
            e.record(st)
            evs.append(e)
        return evs

    def submit(self, q, weights, context_lens, page_table, out_dense, out_sparse):
        """Queue one step on pinned host tensors; returns the step index."""
        i, s = self.n, self.n % 2
        plan = self.plans[s]
        dev = plan.logits.device
        host_in = (q, weights, context_lens, page_table)
        if self.inputs[s] is None:
            self.inputs[s] = [torch.empty(t.shape, dtype=t.dtype, device=dev) for t in host_in]
        dq, dw, dc, dp = self.inputs[s]
        with torch.cuda.stream(self.s_in):
            if self.step_done[s] is not None:
                self.s_in.wait_event(self.step_done[s])
            for d, h in zip(self.inputs[s], host_in):
                d.copy_(h, non_blocking=True)
            in_ready = torch.cuda.Event()
            in_ready.record(self.s_in)
        with torch.cuda.stream(self.s_compute):
            self.s_compute.wait_event(in_ready)
            if self.out_done[s] is not None:
                self.s_compute.wait_event(self.out_done[s])
            dense, sparse = plan.step(dq, self.kv, self.kscale, dw, dp, dc)
            done = torch.cuda.Event()
            done.record(self.s_compute)
        with torch.cuda.stream(self.s_out):
            self.s_out.wait_event(done)
            out_dense.copy_(dense, non_blocking=True)
            out_sparse.copy_(sparse, non_blocking=True)
            oe = torch.cuda.Event()
            oe.record(self.s_out)
        self.step_done[s], self.out_done[s] = done, oe
        self.pending[i] = oe
        self.n += 1
        return i

    def wait(self, i):
        """Block until step i's host outputs are written."""
        self.pending.pop(i).synchronize()

    def synchronize(self):
        for st in (self.s_in, self.s_compute, self.s_out):
            st.synchronize()
        self.pending.clear()
