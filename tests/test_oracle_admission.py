"""Pins for the admission-credit rule and the continuous-batching simulation.

Expected values below are worked out by hand from the rule (credit =
L * ceil((prompt + new - 1) / 16) pages; FIFO; reject if credit > pool).
"""
import numpy as np

import workloads as W
from oracle import admission as A


def test_credit_hand_values():
    assert A.credit_pages(10, 7, 2) == 2          # 16 tokens -> 1 page x 2 layers
    assert A.credit_pages(16, 1, 2) == 2          # 16 tokens -> 1 page
    assert A.credit_pages(17, 1, 2) == 4          # 17 tokens -> 2 pages
    assert A.credit_pages(30, 129, 2) == 20       # 158 tokens -> 10 pages
    assert A.credit_pages(1920, 129, 16) == 16 * 128
    assert A.credit_pages(300, 129, 16) == 16 * 27


def test_scheduler_hand_sequence():
    s = A.Scheduler(num_pages=20, num_layers=2, max_blocks=10, max_slots=4)
    assert s.submit(10, 7) == (s.OK, 0)          # credit 2
    assert s.submit(30, 129) == (s.OK, 1)        # credit 20 (the whole pool)
    assert s.submit(1, 1) == (s.OK, 2)           # credit 2
    assert s.submit(200, 1) == (s.TOO_LARGE, -1)  # 13 pages per layer > 10 blocks
    assert s.submit(40, 129) == (s.TOO_LARGE, -1)  # credit 22 > 20 pages
    assert s.admit() == [0]                      # request 1 needs 20 > 18 free: blocks
    assert s.grow(0, 10) == s.OK
    assert s.events == [(0, 0, 0, 0), (0, 1, 0, 1)]
    assert s.admit() == []                       # FIFO: 2 waits behind 1
    assert s.grow(0, 17) == s.EXHAUSTED          # would exceed its own credit
    assert s.finish(0) == s.OK                   # pushes 0 then 1
    assert s.admit() == [1]                      # slot 0 reused
    assert s.req[1]["slot"] == 0
    assert s.grow(1, 30) == s.OK
    assert s.events[2:] == [(1, 0, 0, 1), (1, 0, 1, 0), (1, 1, 0, 2), (1, 1, 1, 3)]
    assert s.block_table_row(1, 1)[:3] == [2, 3, -1]
    assert s.admit() == []                       # 2 needs 2 pages, 0 unreserved
    assert s.finish(1) == s.OK
    assert s.admit() == [2]


def test_simulation_invariants():
    case = W.case_continuous()
    ids, log, sch = A.simulate(case.prompt_lens, case.decode_steps, case.num_pages, case.num_layers)
    assert all(st == A.Scheduler.OK for st, _ in ids)
    # every request runs exactly decode_steps steps and lengths grow by one per step
    steps = {}
    order = []
    for e in log:
        order += e["admitted"]
        for rid, n in zip(e["running"], e["lens"]):
            steps[rid] = steps.get(rid, 0) + 1
            assert n == case.prompt_lens[rid] + steps[rid]
    assert order == list(range(len(case.prompt_lens)))          # FIFO admission
    assert all(v == case.decode_steps for v in steps.values())
    # no page is ever held by two requests at once; pool capacity respected
    owner = {}
    for rid, layer, j, page in sch.events:
        owner.setdefault(page, []).append(rid)
    assert len(sch.free) == case.num_pages                      # everything returned
    held_peak = max(sum(-(-n // 16) for n in e["lens"]) * case.num_layers for e in log)
    assert held_peak <= case.num_pages
    # continuous batching really overlaps requests
    assert max(len(e["running"]) for e in log) > 1


def test_simulation_pages_disjoint_over_time():
    prompts = np.array([30, 5, 100, 17, 64])
    ids, log, sch = A.simulate(prompts, 20, num_pages=60, num_layers=2)
    live = {}
    held = {}
    # replay events per step boundary: a page must be released before reuse
    for rid, layer, j, page in sch.events:
        held.setdefault(rid, set()).add(page)
    for e in log:
        for rid in e["running"]:
            live[rid] = held[rid]
        running_sets = [held[r] for r in e["running"]]
        allp = [p for st in running_sets for p in st]
        assert len(allp) == len(set(allp))


def test_static_batching_waits_for_the_group():
    """Hand-worked: pool of 20 pages, 2 layers; requests of credit 6, 6, 4
    (prompt + new - 1 = 48 / 48 / 32 tokens -> 3 / 3 / 2 pages per layer).
    All three fit at once; a fourth of credit 6 does not (16 + 6 > 20).
    Continuous admits the fourth as soon as one of the first three frees
    its pages; static waits until all three have finished."""
    for mode, expect_after_one in ((A.Scheduler.CONTINUOUS, [3]), (A.Scheduler.STATIC, [])):
        s = A.Scheduler(num_pages=20, num_layers=2, max_blocks=10, max_slots=8, mode=mode)
        for prompt, new in ((40, 9), (40, 9), (30, 3), (40, 9)):
            assert s.submit(prompt, new)[0] == s.OK
        assert s.admit() == [0, 1, 2]                # credits 6 + 6 + 4 = 16 <= 20
        assert s.admit() == []                        # 6 > 20 - 16
        assert s.finish(2) == s.OK                    # 4 pages of credit come back
        assert s.admit() == expect_after_one          # 6 <= 20 - 12 only for continuous
        if mode == A.Scheduler.STATIC:
            assert s.finish(0) == s.OK
            assert s.admit() == []                    # request 1 still running
            assert s.finish(1) == s.OK
            assert s.admit() == [3]                   # the group has finished


def test_static_simulation_groups_do_not_overlap():
    case = W.case_continuous()
    ids, log, _ = A.simulate(case.prompt_lens, case.decode_steps, case.num_pages,
                             case.num_layers, mode=A.Scheduler.STATIC)
    assert all(st == A.Scheduler.OK for st, _ in ids)
    running = set()
    for e in log:
        if e["admitted"]:
            assert not (running - set(e["admitted"])), "admitted while a group was running"
        running |= set(e["admitted"])
        running -= set(e["finished"])
    admitted = [r for e in log for r in e["admitted"]]
    assert admitted == sorted(admitted) and len(admitted) == len(case.prompt_lens)
