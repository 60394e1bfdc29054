"""Continuous batching over the paged pool: admission credit, on-demand pages,
prompt appends and decode steps, driving the C++ scheduler and the kernels.

From the samir-vllm article, section "Gestion de la KV cache et strategies de
batching": requests are admitted as soon as their page budget is available
(credit = prompt + allowed_new - 1 tokens rounded up to 16-token pages, per
layer), oversize requests are rejected, the prompt fills its pages at
admission and every decode step appends one token per running sequence at its
absolute position and attends over the sequence's own pages.

The scheduler decides admissions and page ids (host C++).  Prompt appends
use per-slot block tables on the device ([L][max_slots][max_blocks]); a decode
step's lengths and tables are packed by the scheduler into one pinned host
block and reach the device in one copy, issued together with the step's
launches by one native call (paged_gqa_decode_append_layers).  The caller supplies
the new K/V/q values through callbacks, so any model (or a synthetic source)
can drive it.  Nothing here computes attention: every token goes through
kv_append_rope / paged_gqa_decode / paged_gqa_decode_append(_layers), or
their INT8-page forms when the pool is an INT8 pool.
"""
from __future__ import annotations

from typing import NamedTuple

import numpy as np
import torch

from . import (HEAD_DIM, NUM_KV_HEADS, NUM_Q_HEADS, OK, PAGE_TOKENS, PkvError, Scheduler,
               alloc_workspace, kv_append_rope, kv_append_rope_int8, kv_append_rope_layers,
               paged_gqa_decode,
               paged_gqa_decode_append_layers, paged_gqa_decode_int8, pkv_read_device_error,
               ERR_REQUEST_TOO_LARGE)


class StepBatch(NamedTuple):
    """One decode step's batch, from ContinuousBatcher.prepare_step."""
    ids: list                 # running request ids, in batch-row order
    lens_h: np.ndarray        # [B] int32 lengths after the step (host)
    lens: torch.Tensor        # the same on the device (a view of dev_block)
    tables: torch.Tensor      # [L, B, P] int32 block tables (a view of dev_block)
    host_block: torch.Tensor  # the packed step block (pinned host memory)
    dev_block: torch.Tensor   # its device copy, written by launch_step
    turn: int                 # which of the two host blocks it is


class ContinuousBatcher:
    """FIFO continuous batching of decode requests on one device.

    pool:        [num_pages, 2, 8, 16, 64] bf16 (one layer per page), or an
                 INT8 pool [num_pages, 8, 2176] uint8 (see new_int8_pool)
    rope_cos/sin [max_pos, 32] fp32 device tables
    fused:       decode steps as one fused append+decode kernel per layer
                 (else kv_append_rope followed by paged_gqa_decode)
    static:      static batching: a new group is admitted only once every
                 request of the current one has finished
    """

    def __init__(self, pool, num_layers, rope_cos, rope_sin, scale, max_blocks=128,
                 max_slots=256, fused=True, static=False):
        self.pool = pool
        self.int8 = pool.dtype == torch.uint8
        self.dev = pool.device
        self.L = num_layers
        self.M = max_blocks
        self.cos, self.sin = rope_cos, rope_sin
        self.scale = float(scale)
        self.fused = fused
        self.sched = Scheduler(pool.shape[0], num_layers, max_blocks, max_slots, static=static)
        self.max_slots = max_slots
        self.tables = torch.full((num_layers, max_slots, max_blocks), -1, dtype=torch.int32,
                                 device=self.dev)
        self.host_tables = np.full((num_layers, max_slots, max_blocks), -1, np.int32)
        self.d_err = torch.zeros(1, dtype=torch.int32, device=self.dev)
        self.workspace = alloc_workspace(max_slots, self.dev)   # serves any batch <= max_slots
        # step blocks (lengths + tables of a step, pkv_sched_pack_step): two
        # pinned host blocks used in turn, each reused only once the copy made
        # from it two steps earlier has run, and one device block
        nmax = self.sched.step_bytes(max_slots, PAGE_TOKENS * max_blocks)
        pin = self.dev.type == "cuda"
        self._host_blocks = [torch.empty(nmax, dtype=torch.uint8, pin_memory=pin) for _ in range(2)]
        self._block_done = [None, None]
        self._block_events = [torch.cuda.Event(), torch.cuda.Event()] if pin else None
        self._turn = 0
        self._dev_block = torch.empty(nmax, dtype=torch.uint8, device=self.dev)
        # prompt appends: positions 0.. and the row index 0 of a one-row table
        # view, for any prompt the tables can hold; a device stage for prompt
        # rows that come from host memory (allocated on first use)
        self._positions = torch.arange(PAGE_TOKENS * max_blocks, dtype=torch.int32, device=self.dev)
        self._row0 = torch.zeros(PAGE_TOKENS * max_blocks, dtype=torch.int32, device=self.dev)
        self._stage = None
        self.prompt = {}           # request id -> prompt tokens
        self.running = []          # request ids in admission order
        self.length = {}           # request id -> KV tokens held
        self.steps_done = {}
        self.slot = {}
        self.rejected = []
        self.uploaded_bytes = 0    # scheduler state copied host -> device so far

    # -- requests -------------------------------------------------------------
    def submit(self, prompt_tokens: int, new_tokens: int):
        """Queue a request; returns its id, or -1 when it can never fit.
        Raises PkvError for an invalid request (fewer than one prompt or new
        token)."""
        st, rid = self.sched.submit(prompt_tokens, new_tokens)
        if st == ERR_REQUEST_TOO_LARGE:
            self.rejected.append((prompt_tokens, new_tokens))
            return -1
        self.prompt[rid] = int(prompt_tokens)
        return rid

    def _upload(self, a: np.ndarray) -> torch.Tensor:
        """Host array -> device tensor without waiting for the device (pinned
        staging; the host allocator keeps the staging block until the copy
        has run)."""
        t = torch.from_numpy(np.ascontiguousarray(a))
        self.uploaded_bytes += t.numel() * t.element_size()
        if self.dev.type == "cuda":
            t = t.pin_memory()
        return t.to(self.dev, non_blocking=True)

    def _sync_rows(self, rid):
        """Copy a request's block-table rows (all layers) to the device."""
        s = self.slot[rid]
        for l in range(self.L):
            row, _ = self.sched.block_table(rid, l)
            self.host_tables[l, s] = row
        self.tables[:, s].copy_(self._upload(self.host_tables[:, s]))

    def admit(self, prompt_kv):
        """Admit what fits and write the prompts' K/V.

        prompt_kv(rid, layer) -> (k [P, 8, 64], v [P, 8, 64]) bf16 tensors
        (host tensors are copied without waiting: a pinned one must stay
        unchanged until the copy has run).  Returns the admitted request ids.
        """
        admitted = self.sched.admit()
        for rid in admitted:
            P = self.prompt[rid]
            if self.sched.grow(rid, P) != OK:
                raise PkvError(7, "ContinuousBatcher.admit")
            _, self.slot[rid] = self.sched.block_table(rid, 0)
            self._sync_rows(rid)
            ks, vs = zip(*(prompt_kv(rid, l) for l in range(self.L)))
            # one native call for every layer: host rows go through the stage
            stage = None
            if ks[0].device != self.dev:
                need = 2 * P * NUM_KV_HEADS * HEAD_DIM * 2
                if self._stage is None or self._stage.numel() < need:
                    self._stage = torch.empty(2 * PAGE_TOKENS * self.M * NUM_KV_HEADS * HEAD_DIM * 2,
                                              dtype=torch.uint8, device=self.dev)
                stage = self._stage
            s = self.slot[rid]
            kv_append_rope_layers(ks, vs, self._positions[:P], self.tables[:, s:s + 1], self.pool,
                                  self.cos, self.sin, token_seq=self._row0[:P], stage=stage,
                                  d_err=self.d_err)
            self.length[rid] = P
            self.steps_done[rid] = 0
        self.running += admitted
        return admitted

    def prepare_step(self) -> "StepBatch":
        """Host side of one decode step for every running request.

        The scheduler grows each request by one token (a new page in every
        layer where its position starts one) and packs the batch's lengths
        (after the step) and block tables [L, B, P] into a pinned host block
        (two C calls); launch_step copies it to the device.  The returned
        batch is consumed by exactly one launch_step; nothing here launches a
        kernel.
        """
        ids_a, lens_h = self.sched.begin_step()
        ids = [int(r) for r in ids_a]
        if ids != self.running:
            raise PkvError(1, "ContinuousBatcher.prepare_step")   # scheduler and batcher disagree
        B = len(ids)
        max_len = int(lens_h.max()) if B else 0
        nbytes = self.sched.step_bytes(B, max_len)
        turn = self._turn
        self._turn ^= 1
        if self._block_done[turn] is not None:
            self._block_done[turn].synchronize()   # its copy from two steps ago has run
        host = self._host_blocks[turn][:nbytes]
        P = self.sched.pack_step(ids_a, max_len, host)
        dev = self._dev_block[:nbytes]
        off = (4 * B + 15) // 16 * 16
        lens = dev[:4 * B].view(torch.int32)
        tables = dev[off:off + 4 * self.L * B * P].view(torch.int32).view(self.L, B, P)
        self.uploaded_bytes += nbytes
        for rid, n in zip(ids, lens_h):
            self.length[rid] = int(n)
            self.steps_done[rid] += 1
        return StepBatch(ids, lens_h, lens, tables, host, dev, turn)

    def _block_sent(self, batch):
        """Mark (on the stream) the point after which the batch's host block may be reused."""
        if self._block_events is not None:
            ev = self._block_events[batch.turn]
            ev.record()
            self._block_done[batch.turn] = ev

    def launch_step(self, batch: "StepBatch", q, k, v, out=None):
        """Device side of one decode step: every layer appends each request's
        new token at its position and attends over the request's pages.

        q [L, B, 32, 64] (un-rotated), k / v [L, B, 8, 64] bf16 device
        tensors, rows in batch.ids order.  Returns out [L, B, 32, 64] bf16.
        Launches kernels only (one fused kernel per layer, or an append and
        a decode): no host synchronisation.
        """
        B = len(batch.ids)
        shapes = ((q, NUM_Q_HEADS), (k, NUM_KV_HEADS), (v, NUM_KV_HEADS))
        for t, h in shapes:
            if tuple(t.shape) != (self.L, B, h, HEAD_DIM):
                raise ValueError(f"expected [{self.L}, {B}, {h}, {HEAD_DIM}], got {tuple(t.shape)}")
            if t.dtype != torch.bfloat16 or t.device != self.dev or not t.is_contiguous():
                raise TypeError("q / k / v must be contiguous bf16 tensors on the pool's device")
        if out is None:
            out = torch.empty((self.L, B, NUM_Q_HEADS, HEAD_DIM), dtype=torch.bfloat16,
                              device=self.dev)
        elif (tuple(out.shape) != (self.L, B, NUM_Q_HEADS, HEAD_DIM) or out.dtype != torch.bfloat16
              or out.device != self.dev or not out.is_contiguous()):
            raise ValueError("out must be a contiguous bf16 [L, B, 32, 64] tensor on the pool's device")
        if B == 0:
            return out
        ms = int(batch.lens_h.max())
        ws = self.workspace
        if self.fused:
            # one C call: the step block's copy, then the L fused launches
            # (layers >= 1 stage their pages while the previous layer ends);
            # the shapes were checked above and the other tensors are the
            # batcher's own, so the binding's per-call checks are skipped
            paged_gqa_decode_append_layers(q, k, v, self.pool, batch.tables, batch.lens, out,
                                           self.cos, self.sin, self.scale, ws, max_seq_len=ms,
                                           d_err=self.d_err, early_kv=1,
                                           host_stage=batch.host_block, dev_stage=batch.dev_block,
                                           check=False)
            self._block_sent(batch)
            return out
        batch.dev_block.copy_(batch.host_block, non_blocking=True)
        self._block_sent(batch)
        positions = batch.lens - 1
        append = kv_append_rope_int8 if self.int8 else kv_append_rope
        decode = paged_gqa_decode_int8 if self.int8 else paged_gqa_decode
        for l in range(self.L):
            bt = batch.tables[l]
            q_rot = torch.empty_like(q[l])
            append(k[l], v[l], positions, bt, self.pool, self.cos, self.sin, q_in=q[l],
                   q_out=q_rot, d_err=self.d_err)
            decode(q_rot, self.pool, bt, batch.lens, out[l], self.scale, workspace=ws,
                   max_seq_len=ms, d_err=self.d_err)
        return out

    def step(self, token_kv, token_q):
        """One decode step for every running request, inputs from callbacks.

        token_kv(rid, layer, pos) -> (k [8, 64], v [8, 64]); token_q(rid, layer,
        pos) -> q [32, 64] (un-rotated).  Returns (running ids, lengths after
        the step, outputs [L, B, 32, 64] bf16 on the device).
        """
        batch = self.prepare_step()
        if not batch.ids:
            return [], batch.lens_h, torch.empty((self.L, 0, NUM_Q_HEADS, HEAD_DIM),
                                                 dtype=torch.bfloat16, device=self.dev)
        pos = [int(p) for p in batch.lens_h - 1]
        qs, ks, vs = [], [], []
        for l in range(self.L):
            qs.append(torch.stack([token_q(r, l, p) for r, p in zip(batch.ids, pos)]))
            kv = [token_kv(r, l, p) for r, p in zip(batch.ids, pos)]
            ks.append(torch.stack([a for a, _ in kv]))
            vs.append(torch.stack([b for _, b in kv]))
        q, k, v = (torch.stack(x).to(self.dev) for x in (qs, ks, vs))
        return batch.ids, batch.lens_h, self.launch_step(batch, q, k, v)

    def retire(self, decode_steps: int):
        """Finish requests that have done `decode_steps` steps; frees their pages."""
        done = [r for r in self.running if self.steps_done[r] == decode_steps]
        for rid in done:
            self.sched.finish(rid)
            s = self.slot.pop(rid)
            self.host_tables[:, s] = -1
            self.tables[:, s] = -1
        self.running = [r for r in self.running if r not in done]
        return done

    def error(self) -> int:
        return pkv_read_device_error(self.d_err)
