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

from . import (OUT_F16, Workspace, coarse_hist_topk, coarse_hist_topk_batch, decode_step,
               decode_step_args,
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
        CUDA events) brackets individual launches for per-kernel timing.
        Without events, the plan's usual shape (the table written by the select
        launch) runs as one library call (``dsa_decode_step``) whose argument
        block is built once per set of input tensors."""
        nn, ws = self.next_n, self.ws
        if events is None and self.fused_table:
            key = tuple((t.data_ptr(), tuple(t.shape), t.dtype)
                        for t in (q, kv, kscale, weights, page_table, context_lens))
            if getattr(self, "_step_key", None) != key:
                self._step_args = decode_step_args(
                    q, kv, kscale, weights, page_table, context_lens, nn, self.k, self.kb,
                    self.logits, self.hist, self.topk_idx, self.block_ids, self.phys,
                    self.valid_lens, self.sparse, self.sparse_idx)
                self._step_key = key
            decode_step(self._step_args, ws)
            return self.topk_idx, self.sparse_idx

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
    """Decode steps fed from and returned to pinned host memory, two in
    flight: while one step computes, the next one's inputs travel in and the
    previous one's results travel out.

    Two slots alternate, each with its own ``DecodePlan``, device copy of the
    per-step inputs (q, weights, context lengths, page table) and stream.  A
    slot's step -- the host-to-device copies, the plan's kernels and the
    device-to-host copies of both index sets -- is captured once as a CUDA
    graph (its first submit runs the step eagerly and captures it), so a
    submit is one graph launch.  A graph holds the addresses of the host
    tensors it was captured with: pass each slot the same pinned tensors on
    every submit and rewrite their contents in place (a slot given other
    tensors is captured again).  The K cache (``kv``, ``kscale``) is resident
    device state that both slots read.  Host inputs may be rewritten, and host
    outputs read, once ``wait(i)`` for the slot's last step has returned.  The
    kernels and the results are those of ``DecodePlan.step``."""

    def __init__(self, B, next_n, max_context, page_size, kv, kscale, k=2048, kb=512,
                 device="cuda"):
        dev = torch.device(device)
        self.device = dev
        self.plans = [DecodePlan(B, next_n, max_context, page_size, k=k, kb=kb, two_level=True,
                                 device=dev) for _ in range(2)]
        self.kv, self.kscale = kv, kscale
        self.streams = [torch.cuda.Stream(device=dev) for _ in range(2)]
        self.inputs = [None, None]
        self.graphs = [None, None]
        self.bound = [None, None]   # host tensor addresses each slot's graph holds
        self.pending = {}           # step index -> event after its host outputs
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
        for st in self.streams:
            st.wait_event(event)

    def record_all(self):
        """An event on each slot's stream, after everything submitted so far."""
        evs = []
        for st in self.streams:
            e = torch.cuda.Event()
            e.record(st)
            evs.append(e)
        return evs

    def _run(self, s, host):
        plan, (dq, dw, dc, dp) = self.plans[s], self.inputs[s]
        for d, h in zip((dq, dw, dc, dp), host[:4]):
            d.copy_(h, non_blocking=True)
        dense, sparse = plan.step(dq, self.kv, self.kscale, dw, dp, dc)
        host[4].copy_(dense, non_blocking=True)
        host[5].copy_(sparse, non_blocking=True)

    def submit(self, q, weights, context_lens, page_table, out_dense, out_sparse):
        """Queue one step on pinned host tensors; returns the step index."""
        i, s = self.n, self.n % 2
        host = (q, weights, context_lens, page_table, out_dense, out_sparse)
        st = self.streams[s]
        key = tuple((t.data_ptr(), tuple(t.shape), t.dtype) for t in host)
        if self.bound[s] != key:
            if not all(t.is_pinned() for t in host):
                raise ValueError("HostStepPipeline needs pinned host tensors")
            if self.inputs[s] is None:
                self.inputs[s] = [torch.empty(t.shape, dtype=t.dtype, device=self.device)
                                  for t in host[:4]]
            with torch.cuda.stream(st):
                self._run(s, host)  # this step, eagerly (sets the kernels' attributes)
            st.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                self._run(s, host)
            self.graphs[s], self.bound[s] = g, key
        else:
            with torch.cuda.stream(st):
                self.graphs[s].replay()
        ev = torch.cuda.Event()
        ev.record(st)
        self.pending[i] = ev
        self.n += 1
        return i

    def wait(self, i):
        """Block until step i's host outputs are written."""
        self.pending.pop(i).synchronize()

    def synchronize(self):
        for st in self.streams:
            st.synchronize()
        self.pending.clear()
