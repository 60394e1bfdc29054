"""C-ABI checks that need no GPU: the library loads, exports every symbol that
include/pkv.h declares, rejects bad arguments before launching anything, and
its host-side RoPE tables and scheduler agree with the FP64 oracle exactly."""
import ctypes
import os
import re
import subprocess
import sys

import numpy as np
import pytest

from paged_kv_gqa_append_gb300 import build as B

B.build()  # no-op when libpkv.so is up to date
import paged_kv_gqa_append_gb300 as pkv  # noqa: E402
import workloads as W  # noqa: E402
from oracle import admission as A, rope  # noqa: E402

HEADER = os.path.join(B.ROOT, "include", "pkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)
    keywords = {"if", "sizeof", "return", "defined"}
    return sorted({n for n in names if n not in keywords and not n.startswith("__")})


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert "kv_append_rope" in names and "paged_gqa_decode" in names
    missing = [n for n in names if not hasattr(pkv.lib, n)]
    assert not missing, missing


def test_int8_page_format_agrees_with_the_oracle():
    # the header's INT8 block, the binding's and the oracle's byte layout
    text = open(HEADER).read()
    m = re.search(r"#define PKV_I8_BLOCK_BYTES .*?/\* (\d+) \*/", text)
    assert m and int(m.group(1)) == 2176
    from oracle import int8_kv as OI
    assert pkv.I8_BLOCK_BYTES == OI.BLOCK_BYTES == W.I8_BLOCK_BYTES == 2176


def test_status_strings():
    assert pkv.status_string(0) == "PKV_OK"
    assert pkv.status_string(6) == "PKV_ERR_DEVICE_INDEX"
    assert pkv.status_string(99) == "PKV_ERR_UNKNOWN"
    assert pkv.lib.pkv_version() >= 100


def test_inv_freq_bit_exact_vs_oracle():
    assert np.array_equal(pkv.pkv_rope_inv_freq_plain(500000.0), rope.inv_freq_plain(500000.0))
    assert np.array_equal(pkv.pkv_rope_inv_freq_plain(10000.0), rope.inv_freq_plain(10000.0))
    assert np.array_equal(pkv.pkv_rope_inv_freq_llama3(), rope.inv_freq_llama3())


def test_rope_table_bit_exact_vs_oracle():
    f = rope.inv_freq_llama3()
    cos_c, sin_c = pkv.pkv_rope_table_fill(pkv.pkv_rope_inv_freq_llama3(), 2048)
    cos_o, sin_o = rope.table(f, 2048)
    assert np.array_equal(cos_c.view(np.uint32), cos_o.view(np.uint32))
    assert np.array_equal(sin_c.view(np.uint32), sin_o.view(np.uint32))


def test_credit_matches_oracle():
    for p, n, l in [(10, 7, 2), (16, 1, 2), (17, 1, 2), (30, 129, 2), (1920, 129, 16), (1, 1, 16)]:
        assert pkv.pkv_credit_pages(p, n, l) == A.credit_pages(p, n, l)


def test_host_side_validation_returns_before_launch():
    """The checks below pass made-up device addresses: they run in a child
    process that sees no GPU (CUDA_VISIBLE_DEVICES empty), so even a check
    that let one through could never launch a kernel on them."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    code = "import tests.test_abi_cpu as t; t._host_validation_checks()"
    r = subprocess.run([sys.executable, "-c", code], cwd=B.ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr


def _host_validation_checks():
    import torch
    assert not torch.cuda.is_available()
    L = pkv.lib
    null = None
    # append: null pointers, bad sizes
    assert L.kv_append_rope(null, null, null, null, 4, null, 1, 128, 128, null, 8, null, null,
                            2048, null, null, null, null) == 1
    assert L.kv_append_rope(null, null, null, null, -1, null, 1, 128, 128, null, 8, null, null,
                            2048, null, null, null, null) == 1
    assert L.kv_append_rope(null, null, null, null, 0, null, 1, 128, 128, null, 8, null, null,
                            2048, null, null, null, null) == 0      # nothing to do
    # append: q_in without q_out
    fake = ctypes.c_void_p(0x10000)
    assert L.kv_append_rope(fake, fake, fake, null, 1, fake, 1, 128, 128, fake, 8, fake, fake,
                            2048, fake, null, null, null) == 1
    # append: misaligned k
    odd = ctypes.c_void_p(0x10002)
    assert L.kv_append_rope(odd, fake, fake, null, 1, fake, 1, 128, 128, fake, 8, fake, fake,
                            2048, null, null, null, null) == 2
    # decode: zero sequences is a no-op; nulls; stride < max_blocks; misaligned pool
    assert L.paged_gqa_decode(null, null, 8, null, 128, 128, null, 0, 0, null, 0.125, null, 0,
                              null, null) == 0
    assert L.paged_gqa_decode(null, null, 8, null, 128, 128, null, 1, 16, null, 0.125, null, 0,
                              null, null) == 1
    assert L.paged_gqa_decode(fake, fake, 8, fake, 64, 128, fake, 1, 16, fake, 0.125, fake, 1 << 20,
                              null, null) == 1
    assert L.paged_gqa_decode(fake, odd, 8, fake, 128, 128, fake, 1, 16, fake, 0.125, fake, 1 << 20,
                              null, null) == 2
    assert L.paged_gqa_decode(fake, fake, 8, fake, 128, 128, fake, 5000, 16, fake, 0.125, fake,
                              1 << 30, null, null) == 3
    assert L.paged_gqa_decode(fake, fake, 8, fake, 128, 128, fake, 1, 16, fake, float("nan"), fake,
                              1 << 20, null, null) == 1
    # allocation-free decode: the same checks, all before any device work
    NA = L.paged_gqa_decode_noalloc
    assert NA(null, null, 8, null, 128, 128, null, 0, 0, null, 0.125, null, null) == 0
    assert NA(null, fake, 8, fake, 128, 128, fake, 1, 16, fake, 0.125, null, null) == 1
    assert NA(fake, fake, 8, fake, 64, 128, fake, 1, 16, fake, 0.125, null, null) == 1
    assert NA(fake, odd, 8, fake, 128, 128, fake, 1, 16, fake, 0.125, null, null) == 2
    assert NA(fake, fake, 8, fake, 128, 128, fake, 1, 16, fake, float("nan"), null, null) == 1
    assert NA(fake, fake, 8, fake, 128, 128, fake, 5000, 16, fake, 0.125, null, null) == 3
    # prefill: nothing to do; nulls; stride < max_blocks; misaligned q; NaN scale; too many seqs
    PF = L.paged_gqa_prefill
    assert PF(null, 0, null, null, 8, null, 128, 128, null, 0, 16, null, 0.125, null, null) == 0
    assert PF(null, 16, null, null, 8, null, 128, 128, null, 1, 16, null, 0.125, null, null) == 1
    assert PF(fake, 16, fake, fake, 8, fake, 64, 128, fake, 1, 16, fake, 0.125, null, null) == 1
    assert PF(odd, 16, fake, fake, 8, fake, 128, 128, fake, 1, 16, fake, 0.125, null, null) == 2
    assert PF(fake, 16, fake, fake, 8, fake, 128, 128, fake, 1, 16, fake, float("nan"), null,
              null) == 1
    assert PF(fake, 16, fake, fake, 8, fake, 128, 128, fake, 70000, 16, fake, 0.125, null,
              null) == 3
    # argmax: nothing to do; bad sizes; nulls; misaligned
    AM = L.pkv_argmax_f32
    assert AM(null, 0, 10, 10, null, null) == 0
    assert AM(fake, 4, 0, 10, fake, null) == 1
    assert AM(fake, 4, 10, 9, fake, null) == 1
    assert AM(null, 4, 10, 10, fake, null) == 1
    assert AM(ctypes.c_void_p(0x10001), 4, 10, 10, fake, null) == 2
    # INT8 append: nothing to do; null pool; misaligned pool
    A8 = L.kv_append_rope_int8
    assert A8(null, null, null, null, 0, null, 1, 128, 128, null, 8, null, null, 2048, null, null,
              null, null) == 0
    assert A8(fake, fake, fake, null, 1, fake, 1, 128, 128, null, 8, fake, fake, 2048, null, null,
              null, null) == 1
    assert A8(fake, fake, fake, null, 1, fake, 1, 128, 128, ctypes.c_void_p(0x10004), 8, fake, fake,
              2048, null, null, null, null) == 2
    # layered append: nothing to do; a null layer entry; a missing, short or
    # misaligned stage for host rows; a layer stride below one table; a
    # misaligned device row; a misaligned INT8 pool -- all refused before any
    # CUDA call (this process has no GPU, so a CUDA call would fail with 5)
    AL = L.kv_append_rope_layers
    arr = lambda *xs: (ctypes.c_void_p * len(xs))(*xs)
    two = arr(fake, fake)
    def al(k=two, v=two, n=2, host=0, stage=null, stage_bytes=0, T=4, bt_ls=1 << 16, pool=fake,
           int8=0):
        return AL(k, v, n, host, stage, stage_bytes, fake, null, T, fake, bt_ls, 1, 128, 128, pool,
                  8, int8, fake, fake, 2048, null, null)
    assert al(n=0) == 0 and al(T=0) == 0
    assert al(k=arr(fake, null)) == 1
    assert al(host=1) == 1
    assert al(host=1, stage=fake, stage_bytes=2 * 4 * 1024 - 16) == 1
    assert al(host=1, stage=ctypes.c_void_p(0x10008), stage_bytes=1 << 20) == 2
    assert al(bt_ls=100) == 1
    assert al(v=arr(fake, odd)) == 2
    assert al(pool=ctypes.c_void_p(0x10004), int8=1) == 2
    assert al(int8=2) == 1
    # INT8 decode: nothing to do; null pool; misaligned pool; bad option sets
    D8 = L.paged_gqa_decode_int8
    assert D8(null, null, 8, null, 128, 128, null, 0, 0, null, 0.125, null, 0, null, null) == 0
    assert D8(fake, null, 8, fake, 128, 128, fake, 1, 16, fake, 0.125, fake, 1 << 20, null,
              null) == 1
    assert D8(fake, ctypes.c_void_p(0x10008), 8, fake, 128, 128, fake, 1, 16, fake, 0.125, fake,
              1 << 20, null, null) == 2
    for bad in (pkv.DecodeOpts(pkv.COMPUTE_FMA, 0, 0, 0, 0, 0, 0, 0),
                pkv.DecodeOpts(pkv.COMPUTE_TENSOR, 0, 0, 3, 16, 0, 0, 0),
                pkv.DecodeOpts(pkv.COMPUTE_TENSOR, 0, 0, 0, 0, 1, 0, 0),
                pkv.DecodeOpts(pkv.COMPUTE_TENSOR, 0, 0, 0, 0, 0, 1, 0)):
        assert L.paged_gqa_decode_int8_ex(fake, fake, 8, fake, 128, 128, fake, 1, 16, fake, 0.125,
                                          fake, 1 << 20, null, null, ctypes.byref(bad)) == 1
    # fused INT8 step: null new token; misaligned pool; a non-default configuration
    F8 = L.paged_gqa_decode_append_int8
    assert F8(fake, null, fake, fake, fake, 2048, fake, 8, fake, 128, 128, fake, 1, 16, null, fake,
              0.125, fake, 1 << 20, null, null, null) == 1
    assert F8(fake, fake, fake, fake, fake, 2048, ctypes.c_void_p(0x10008), 8, fake, 128, 128, fake, 1,
              16, null, fake, 0.125, fake, 1 << 20, null, null, null) == 2
    four = pkv.DecodeOpts(pkv.COMPUTE_TENSOR, 0, 0, 4, 16, 0, 0, 0)
    assert F8(fake, fake, fake, fake, fake, 2048, fake, 8, fake, 128, 128, fake, 1, 16, null, fake,
              0.125, fake, 1 << 20, null, null, ctypes.byref(four)) == 1


def _run_cpp_schedule(case, static=False, begin_step=False):
    """Drive the C++ scheduler with the oracle's step loop; return its log.
    With begin_step, each decode step is one pkv_sched_begin_step call (and
    its packed block is checked against the scheduler's tables) instead of
    one grow per request."""
    s = pkv.Scheduler(case.num_pages, case.num_layers, W.MAX_BLOCKS, 256, static=static)
    ids = [s.submit(int(p), case.allowed_new_tokens) for p in case.prompt_lens]
    running, length, done, log = [], {}, {}, []
    while s.stats()["queued"] or running:
        admitted = s.admit()
        for rid in admitted:
            assert s.grow(rid, int(case.prompt_lens[rid])) == pkv.OK
            length[rid], done[rid] = int(case.prompt_lens[rid]), 0
        running += admitted
        lens = []
        if begin_step:
            b_ids, b_lens = s.begin_step()
            assert b_ids.tolist() == running
            for rid, n in zip(running, b_lens.tolist()):
                assert n == length[rid] + 1
            _check_packed_block(s, b_ids, b_lens, case.num_layers)
        for rid in running:
            if not begin_step:
                assert s.grow(rid, length[rid] + 1) == pkv.OK
            length[rid] += 1
            done[rid] += 1
            lens.append(length[rid])
        finished = [r for r in running if done[r] == case.decode_steps]
        log.append(dict(admitted=admitted, running=list(running), lens=lens, finished=finished))
        for rid in finished:
            s.finish(rid)
        running = [r for r in running if r not in finished]
    return ids, log, s


def _check_packed_block(s, ids, lens, L):
    """The step block pkv_sched_pack_step writes: lengths, then per layer the
    requests' page ids padded with -1 to P = ceil(max length / 16) entries."""
    B = len(ids)
    max_len = int(lens.max()) if B else 0
    n = s.step_bytes(B, max_len)
    block = np.full(n + 16, 0x55, np.uint8)            # 16 guard bytes that must stay untouched
    P = s.pack_step(ids, max_len, block[:n])
    assert P == max(1, -(-max_len // 16)) and (block[n:] == 0x55).all()
    assert block[:4 * B].view(np.int32).tolist() == lens.tolist()
    off = (4 * B + 15) // 16 * 16
    tab = block[off:off + 4 * L * B * P].view(np.int32).reshape(L, B, P)
    for l in range(L):
        for b, rid in enumerate(ids.tolist()):
            row, _ = s.block_table(rid, l)
            assert tab[l, b].tolist() == row[:P].tolist()
    if B:
        with pytest.raises(pkv.PkvError):            # a length above max_len
            s.pack_step(ids, max_len - 1, block[:n])
        with pytest.raises(pkv.PkvError):            # a block too small
            s.pack_step(ids, max_len, block[:n - 4])


@pytest.mark.parametrize("static", [False, True])
@pytest.mark.parametrize("begin_step", [False, True])
def test_scheduler_matches_oracle_on_continuous_mix(static, begin_step):
    case = W.case_continuous()
    ids_o, log_o, sch_o = A.simulate(case.prompt_lens, case.decode_steps, case.num_pages,
                                     case.num_layers,
                                     mode=A.Scheduler.STATIC if static else A.Scheduler.CONTINUOUS)
    ids_c, log_c, sch_c = _run_cpp_schedule(case, static, begin_step)
    assert [r for _, r in ids_c] == [r for _, r in ids_o]
    assert len(log_c) == len(log_o)
    for a, b in zip(log_c, log_o):
        for key in ("admitted", "running", "lens", "finished"):
            assert a[key] == b[key], key
    assert sch_c.events() == sch_o.events
    assert sch_c.stats()["free"] == case.num_pages and sch_c.stats()["reserved"] == 0


def test_scheduler_rejects_and_blocks():
    s = pkv.Scheduler(num_pages=20, num_layers=2, max_blocks=10, max_slots=4)
    assert s.submit(10, 7) == (pkv.OK, 0)
    assert s.submit(30, 129) == (pkv.OK, 1)
    assert s.submit(1, 1) == (pkv.OK, 2)
    assert s.submit(200, 1) == (pkv.ERR_REQUEST_TOO_LARGE, -1)
    assert s.submit(40, 129) == (pkv.ERR_REQUEST_TOO_LARGE, -1)
    assert s.admit() == [0]
    assert s.grow(0, 10) == pkv.OK
    assert s.admit() == []
    assert s.grow(0, 17) == pkv.ERR_POOL_EXHAUSTED
    s.finish(0)
    assert s.admit() == [1]
    assert s.grow(1, 30) == pkv.OK
    assert s.events() == [(0, 0, 0, 0), (0, 1, 0, 1), (1, 0, 0, 1), (1, 0, 1, 0), (1, 1, 0, 2),
                          (1, 1, 1, 3)]
    row, slot = s.block_table(1, 1)
    assert list(row[:3]) == [2, 3, -1] and slot == 0
    assert s.stats() == dict(free=16, reserved=16, queued=1, running=1)


def test_scheduler_misuse_is_refused_without_state_change():
    # the C scheduler's contract for calls out of order or out of range:
    # PKV_ERR_INVALID_ARGUMENT, and nothing allocated or released
    lib, INV = pkv.lib, pkv.ERR_INVALID_ARGUMENT
    i = ctypes.c_int
    assert not lib.pkv_sched_create(0, 2, 8, 4) and not lib.pkv_sched_create(16, 2, 8, 0)
    assert lib.pkv_sched_set_mode(None, 0) == INV
    assert lib.pkv_sched_grow(None, 0, 1) == INV and lib.pkv_sched_finish(None, 0) == INV
    assert lib.pkv_sched_event_count(None) == -1
    s = lib.pkv_sched_create(16, 2, 4, 2)
    assert s
    try:
        rid, n, adm = i(-7), i(-1), (i * 4)()
        assert lib.pkv_sched_set_mode(s, 2) == INV
        assert lib.pkv_sched_submit(s, 0, 5, ctypes.byref(rid)) == INV
        assert lib.pkv_sched_submit(s, 5, 0, ctypes.byref(rid)) == INV
        assert lib.pkv_sched_submit(s, 5, 5, None) == INV
        # 62 + 5 - 1 tokens need 5 pages a layer, past max_blocks 4
        assert lib.pkv_sched_submit(s, 62, 5, ctypes.byref(rid)) == pkv.ERR_REQUEST_TOO_LARGE
        assert rid.value == -1
        assert lib.pkv_sched_submit(s, 20, 5, ctypes.byref(rid)) == pkv.OK and rid.value == 0
        assert lib.pkv_sched_grow(s, 0, 1) == INV      # still queued
        assert lib.pkv_sched_finish(s, 0) == INV       # still queued
        assert lib.pkv_sched_admit(s, None, 4, ctypes.byref(n)) == INV
        assert lib.pkv_sched_admit(s, adm, -1, ctypes.byref(n)) == INV
        assert lib.pkv_sched_admit(s, adm, 4, ctypes.byref(n)) == pkv.OK and n.value == 1
        assert lib.pkv_sched_grow(s, 1, 1) == INV      # unknown id
        assert lib.pkv_sched_grow(s, 0, -1) == INV
        assert lib.pkv_sched_grow(s, 0, 4 * 16 + 1) == INV      # past max_blocks
        assert lib.pkv_sched_grow(s, 0, 20) == pkv.OK
        assert lib.pkv_sched_grow(s, 0, 33) == pkv.ERR_POOL_EXHAUSTED   # past its credit
        # begin_step: room for the batch, then all or nothing at the credit's edge
        bid, blen, nb = (ctypes.c_int32 * 4)(), (ctypes.c_int32 * 4)(), i(-1)
        assert lib.pkv_sched_begin_step(s, bid, blen, 0, ctypes.byref(nb)) == INV
        assert lib.pkv_sched_begin_step(None, bid, blen, 4, ctypes.byref(nb)) == INV
        assert lib.pkv_sched_begin_step(s, bid, blen, 4, ctypes.byref(nb)) == pkv.OK
        assert nb.value == 1 and bid[0] == 0 and blen[0] == 21
        assert lib.pkv_sched_grow(s, 0, 32) == pkv.OK  # the credit's last token
        ev = lib.pkv_sched_event_count(s)
        assert lib.pkv_sched_begin_step(s, bid, blen, 4, ctypes.byref(nb)) == pkv.ERR_POOL_EXHAUSTED
        assert lib.pkv_sched_event_count(s) == ev      # nothing taken
        assert lib.pkv_sched_pack_step(s, bid, 1, 16, None, 0) == INV   # null block
        row = (ctypes.c_int32 * 4)()
        assert lib.pkv_sched_block_table(s, 0, 2, row, None) == INV     # layer out of range
        assert lib.pkv_sched_block_table(s, 0, 1, None, None) == INV
        assert lib.pkv_sched_event(s, lib.pkv_sched_event_count(s), None, None, None, None) == INV
        free = i(0)
        assert lib.pkv_sched_stats(s, ctypes.byref(free), None, None, None) == pkv.OK
        assert free.value == 16 - 4                    # 2 layers x 2 pages taken (the credit)
        assert lib.pkv_sched_finish(s, 0) == pkv.OK
        assert lib.pkv_sched_finish(s, 0) == INV       # finished twice
        assert lib.pkv_sched_grow(s, 0, 1) == INV      # finished
        assert lib.pkv_sched_stats(s, ctypes.byref(free), None, None, None) == pkv.OK
        assert free.value == 16
    finally:
        lib.pkv_sched_destroy(s)


def test_int8_block_format_of_the_kernels_matches_the_oracle(tmp_path):
    """The byte positions the append and decode kernels use (csrc/i8_layout.cuh,
    compiled here for the host) against the oracle's own statement of the
    block format (int8_kv.block_positions), for every code and scale byte, and
    the stored byte of every code."""
    import shutil
    from oracle import int8_kv as OI
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    src = tmp_path / "layout.cpp"
    src.write_text(
        "#include <cstdio>\n#define __host__\n#define __device__\n"
        f'#include "{B.CSRC}/i8_layout.cuh"\n'
        "using namespace pkv;\nint main() {\n"
        "  for (int t = 0; t < 16; ++t) for (int d = 0; d < 64; ++d)\n"
        "    printf(\"%u %u\\n\", i8_k_byte(t, d), i8_v_byte(t, d));\n"
        "  for (int t = 0; t < 16; ++t) printf(\"%u %u\\n\", i8_k_scale_byte(t), i8_v_scale_byte(t));\n"
        "  for (int c = -128; c < 128; ++c) printf(\"%u\\n\", (unsigned)i8_code_byte((signed char)c));\n"
        "  return 0;\n}\n")
    exe = tmp_path / "layout"
    r = subprocess.run([cxx, "-std=c++17", "-O0", str(src), "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    lines = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    kv = np.array([list(map(int, ln.split())) for ln in lines[:1024]])
    sc = np.array([list(map(int, ln.split())) for ln in lines[1024:1040]])
    cb = np.array([int(ln) for ln in lines[1040:1296]])
    k, v, ks, vs = OI.block_positions()
    assert np.array_equal(kv[:, 0].reshape(16, 64), k) and np.array_equal(kv[:, 1].reshape(16, 64), v)
    assert np.array_equal(sc[:, 0], ks) and np.array_equal(sc[:, 1], vs)
    assert np.array_equal(cb, (np.arange(-128, 128) + 128) % 256)   # code + 128 as a byte
