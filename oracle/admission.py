"""Admission credit and continuous batching over a page pool (oracle; tests only).

From the samir-vllm article, "Gestion de la KV cache et strategies de batching":
  * continuous batching admits a request as soon as its page budget is
    available; static batching waits for the current group to finish;
  * the admission credit is prompt_tokens + allowed_new_tokens - 1 tokens,
    rounded up to 16-token pages, for each layer;
  * a request whose budget exceeds the whole pool is rejected with an explicit
    error, so it can never deadlock the queue.
The tiny-vllm chapter ("What else is set up in the initialization block") keeps
a free-page list 0..N-1 and block tables initialised to -1.

Readings where the article is silent (the C++ scheduler follows the same rules):
  * strict FIFO: the head of the queue blocks later requests until it fits;
  * a request fits when credit <= free pages - pages still reserved by the
    running requests (credit minus the pages they already hold);
  * pages are taken on demand, when a sequence first needs a page in a layer
    (prompt pages at admission, one more when a position starts a new page),
    from the top of a LIFO free stack that starts as [N-1, ..., 1, 0] (so page
    0 comes first);
  * a finished request returns its pages layer by layer in logical order,
    pushed onto the stack in that order; its slot (block-table row) is freed;
  * a new request takes the lowest free slot;
  * static batching: no request is admitted while any request of the
    current group is still running; once all have finished, the next group
    is the FIFO prefix admitted by the same fit rule.
"""
from __future__ import annotations

PAGE_TOKENS = 16


def credit_pages(prompt_tokens: int, allowed_new_tokens: int, num_layers: int,
                 page_tokens: int = PAGE_TOKENS) -> int:
    """Pages reserved at admission: L * ceil((prompt + new - 1) / 16)."""
    tokens = prompt_tokens + allowed_new_tokens - 1
    pages_per_layer = -(-tokens // page_tokens) if tokens > 0 else 0
    return num_layers * pages_per_layer


class Scheduler:
    """FIFO admission with credit reservation and on-demand page allocation."""

    OK, EXHAUSTED, TOO_LARGE, INVALID = "ok", "exhausted", "too_large", "invalid"
    CONTINUOUS, STATIC = "continuous", "static"

    def __init__(self, num_pages: int, num_layers: int, max_blocks: int, max_slots: int,
                 mode: str = CONTINUOUS):
        assert mode in (self.CONTINUOUS, self.STATIC)
        self.mode = mode
        self.num_pages = num_pages
        self.num_layers = num_layers
        self.max_blocks = max_blocks
        self.max_slots = max_slots
        self.free = list(range(num_pages - 1, -1, -1))   # pop() -> lowest id first
        self.queue = []                                   # FIFO of request ids
        self.req = {}                                     # id -> dict
        self.slot_owner = [None] * max_slots
        self.next_id = 0
        self.events = []                                  # (rid, layer, logical page, page id)

    # -- bookkeeping -------------------------------------------------------
    def reserved_outstanding(self) -> int:
        return sum(r["credit"] - r["held"] for r in self.req.values() if r["state"] == "running")

    def submit(self, prompt_tokens: int, allowed_new_tokens: int):
        """Queue a request.  Returns (status, id); oversize requests are rejected."""
        c = credit_pages(prompt_tokens, allowed_new_tokens, self.num_layers)
        if prompt_tokens < 1 or allowed_new_tokens < 1:
            return self.INVALID, -1
        if c > self.num_pages or -(-(prompt_tokens + allowed_new_tokens - 1) // PAGE_TOKENS) > self.max_blocks:
            return self.TOO_LARGE, -1
        rid = self.next_id
        self.next_id += 1
        self.req[rid] = dict(prompt=prompt_tokens, new=allowed_new_tokens, credit=c, held=0,
                             state="queued", slot=-1,
                             pages=[[] for _ in range(self.num_layers)])
        self.queue.append(rid)
        return self.OK, rid

    def admit(self):
        """Admit queued requests in FIFO order while the head fits.  Returns ids.

        In static mode nothing is admitted while a request is running."""
        admitted = []
        if self.mode == self.STATIC and any(r["state"] == "running" for r in self.req.values()):
            return admitted
        while self.queue:
            rid = self.queue[0]
            r = self.req[rid]
            if r["credit"] > len(self.free) - self.reserved_outstanding():
                break
            if None not in self.slot_owner:
                break
            slot = self.slot_owner.index(None)
            self.queue.pop(0)
            self.slot_owner[slot] = rid
            r["slot"], r["state"] = slot, "running"
            admitted.append(rid)
        return admitted

    def grow(self, rid: int, new_len: int):
        """Make every layer hold pages for positions [0, new_len)."""
        r = self.req[rid]
        need = -(-new_len // PAGE_TOKENS)
        if r["state"] != "running" or need > self.max_blocks:
            return self.INVALID
        extra = sum(max(0, need - len(r["pages"][l])) for l in range(self.num_layers))
        if r["held"] + extra > r["credit"] or extra > len(self.free):
            return self.EXHAUSTED
        for l in range(self.num_layers):
            while len(r["pages"][l]) < need:
                page = self.free.pop()
                self.events.append((rid, l, len(r["pages"][l]), page))
                r["pages"][l].append(page)
                r["held"] += 1
        return self.OK

    def finish(self, rid: int):
        r = self.req[rid]
        if r["state"] != "running":
            return self.INVALID
        for l in range(self.num_layers):
            for page in r["pages"][l]:
                self.free.append(page)
            r["pages"][l] = []
        r["held"] = 0
        self.slot_owner[r["slot"]] = None
        r["state"], r["slot"] = "done", -1
        return self.OK

    def block_table_row(self, rid: int, layer: int):
        row = [-1] * self.max_blocks
        for j, page in enumerate(self.req[rid]["pages"][layer]):
            row[j] = page
        return row


def simulate(prompt_lens, decode_steps: int, num_pages: int, num_layers: int,
             max_blocks: int = 128, max_slots: int = 256, mode: str = Scheduler.CONTINUOUS):
    """Run the continuous-batching schedule; return the per-step event log.

    Step loop: admit (FIFO) -> allocate prompt pages for the newly admitted ->
    every running request grows by one position and decodes -> requests that
    have done `decode_steps` steps finish and free their pages.
    Each log entry: dict(step, admitted=[ids], running=[ids in admission
    order], lens=[KV length after this step's append], finished=[ids]).
    Returns (submit results, log, scheduler); ``scheduler.events`` lists every
    page allocation as (request, layer, logical page, page id) in order.
    """
    sch = Scheduler(num_pages, num_layers, max_blocks, max_slots, mode)
    ids = []
    for p in prompt_lens:
        st, rid = sch.submit(int(p), decode_steps + 1)
        ids.append((st, rid))
    running, length, done_steps, log = [], {}, {}, []
    step = 0
    while sch.queue or running:
        admitted = sch.admit()
        for rid in admitted:
            assert sch.grow(rid, sch.req[rid]["prompt"]) == sch.OK
            length[rid] = sch.req[rid]["prompt"]
            done_steps[rid] = 0
        running += admitted
        if not running:
            raise RuntimeError("queue head can never be admitted")
        lens = []
        for rid in running:
            assert sch.grow(rid, length[rid] + 1) == sch.OK
            length[rid] += 1
            done_steps[rid] += 1
            lens.append(length[rid])
        finished = [rid for rid in running if done_steps[rid] == decode_steps]
        log.append(dict(step=step, admitted=list(admitted), running=list(running), lens=lens,
                        finished=list(finished)))
        for rid in finished:
            sch.finish(rid)
        running = [rid for rid in running if rid not in finished]
        step += 1
    return ids, log, sch
