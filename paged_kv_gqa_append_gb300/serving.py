"""Continuous batching over the paged pool: admission credit, on-demand pages,
prompt appends and decode steps, driving the C++ scheduler and the kernels.

From the samir-vllm article, section "Gestion de la KV cache et strategies de
batching": requests are admitted as soon as their page budget is available
(credit = prompt + allowed_new - 1 tokens rounded up to 16-token pages, per
layer), oversize requests are rejected, the prompt fills its pages at
admission and every decode step appends one token per running sequence at its
absolute position and attends over the sequence's own pages.

The scheduler decides admissions and page ids (host C++); block tables live
on the device per slot ([L][max_slots][max_blocks]), and each step gathers
the running sequences' rows into a packed batch table.  The caller supplies
the new K/V/q values through callbacks, so any model (or a synthetic source)
can drive it.  Nothing here computes attention: every token goes through
kv_append_rope / paged_gqa_decode(_append), or their INT8-page forms when the
pool is an INT8 pool.
"""
from __future__ import annotations

import numpy as np
import torch

from . import (OK, PAGE_TOKENS, PkvError, Scheduler, alloc_workspace, kv_append_rope,
               kv_append_rope_int8, paged_gqa_decode, paged_gqa_decode_append,
               paged_gqa_decode_append_int8, paged_gqa_decode_int8, pkv_read_device_error,
               ERR_REQUEST_TOO_LARGE)


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
        self.prompt = {}           # request id -> prompt tokens
        self.running = []          # request ids in admission order
        self.length = {}           # request id -> KV tokens held
        self.steps_done = {}
        self.slot = {}
        self.rejected = []

    # -- requests -------------------------------------------------------------
    def submit(self, prompt_tokens: int, new_tokens: int):
        """Queue a request; returns its id, or -1 when it can never fit."""
        st, rid = self.sched.submit(prompt_tokens, new_tokens)
        if st == ERR_REQUEST_TOO_LARGE:
            self.rejected.append((prompt_tokens, new_tokens))
            return -1
        self.prompt[rid] = int(prompt_tokens)
        return rid

    def _sync_rows(self, rid):
        """Copy a request's block-table rows (all layers) to the device."""
        s = self.slot[rid]
        for l in range(self.L):
            row, _ = self.sched.block_table(rid, l)
            self.host_tables[l, s] = row
        self.tables[:, s].copy_(torch.from_numpy(self.host_tables[:, s]))

    def admit(self, prompt_kv):
        """Admit what fits and write the prompts' K/V.

        prompt_kv(rid, layer) -> (k [P, 8, 64], v [P, 8, 64]) bf16 tensors.
        Returns the admitted request ids.
        """
        admitted = self.sched.admit()
        for rid in admitted:
            P = self.prompt[rid]
            if self.sched.grow(rid, P) != OK:
                raise PkvError(7, "ContinuousBatcher.admit")
            _, self.slot[rid] = self.sched.block_table(rid, 0)
            self._sync_rows(rid)
            pos = torch.arange(P, dtype=torch.int32, device=self.dev)
            rows = torch.full((P,), self.slot[rid], dtype=torch.int32, device=self.dev)
            append = kv_append_rope_int8 if self.int8 else kv_append_rope
            for l in range(self.L):
                k, v = prompt_kv(rid, l)
                append(k.to(self.dev), v.to(self.dev), pos, self.tables[l], self.pool,
                       self.cos, self.sin, token_seq=rows, d_err=self.d_err)
            self.length[rid] = P
            self.steps_done[rid] = 0
        self.running += admitted
        return admitted

    def step(self, token_kv, token_q, out_layers=None):
        """One decode step for every running request.

        token_kv(rid, layer, pos) -> (k [8, 64], v [8, 64]); token_q(rid, layer,
        pos) -> q [32, 64] (un-rotated).  Returns (running ids, lengths after
        the step, outputs [L, B, 32, 64] bf16 on the device).
        """
        ids = list(self.running)
        B = len(ids)
        for rid in ids:
            if self.sched.grow(rid, self.length[rid] + 1) != OK:
                raise PkvError(7, "ContinuousBatcher.step")
            if self.length[rid] % PAGE_TOKENS == 0:      # a new page in every layer
                self._sync_rows(rid)
        lens_h = np.array([self.length[r] + 1 for r in ids], np.int32)
        slots = torch.tensor([self.slot[r] for r in ids], dtype=torch.long, device=self.dev)
        lens = torch.from_numpy(lens_h).to(self.dev)
        pos = lens - 1
        out = torch.empty((self.L, B, 32, 64), dtype=torch.bfloat16, device=self.dev)
        ws = self.workspace
        for l in range(self.L):
            q = torch.stack([token_q(r, l, self.length[r]) for r in ids]).to(self.dev)
            kv = [token_kv(r, l, self.length[r]) for r in ids]
            k = torch.stack([a for a, _ in kv]).to(self.dev)
            v = torch.stack([b for _, b in kv]).to(self.dev)
            bt = self.tables[l].index_select(0, slots).contiguous()
            if self.fused:
                step = paged_gqa_decode_append_int8 if self.int8 else paged_gqa_decode_append
                step(q, k, v, self.pool, bt, lens, out[l], self.cos, self.sin, self.scale,
                     workspace=ws, d_err=self.d_err)
            else:
                q_rot = torch.empty_like(q)
                append = kv_append_rope_int8 if self.int8 else kv_append_rope
                decode = paged_gqa_decode_int8 if self.int8 else paged_gqa_decode
                append(k, v, pos, bt, self.pool, self.cos, self.sin, q_in=q, q_out=q_rot,
                       d_err=self.d_err)
                decode(q_rot, self.pool, bt, lens, out[l], self.scale, workspace=ws,
                       d_err=self.d_err)
        for rid in ids:
            self.length[rid] += 1
            self.steps_done[rid] += 1
        return ids, lens_h, out

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
