"""Python binding of libpkv.so: paged GQA decode and fused RoPE + paged KV append.

The functions carry the C-ABI names and only marshal arguments: they check
dtypes, devices and shapes of torch tensors, pass raw pointers, sizes and the
current CUDA stream to the library, and raise ``PkvError`` on a non-zero
status.  Every step of the computation runs in the library's sm_103a kernels;
there is no fallback: the first call raises when libpkv.so is missing (build
it with ``python -m paged_kv_gqa_append_gb300.build``).

Tensor layouts (see include/pkv.h):
    kv_pool       [num_pages, 2, 8, 16, 64] bf16   (K = 0, V = 1), 32 KiB/page
    block_tables  [num_seqs, >= max_blocks] int32  (-1 = no page)
    q / out       [num_seqs, 32, 64] bf16
    k / v         [T, 8, 64] bf16;  positions / token_seq [T] int32
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

NUM_Q_HEADS = 32
NUM_KV_HEADS = 8
HEAD_DIM = 64
PAGE_TOKENS = 16
ROPE_PAIRS = 32

COMPUTE_TENSOR = 0
COMPUTE_FMA = 1
SCHEDULE_STATIC, SCHEDULE_DYNAMIC, SCHEDULE_AUTO = 0, 1, 2

STATUS = {
    0: "PKV_OK", 1: "PKV_ERR_INVALID_ARGUMENT", 2: "PKV_ERR_MISALIGNED",
    3: "PKV_ERR_UNSUPPORTED_SHAPE", 4: "PKV_ERR_WORKSPACE_TOO_SMALL", 5: "PKV_ERR_CUDA",
    6: "PKV_ERR_DEVICE_INDEX", 7: "PKV_ERR_POOL_EXHAUSTED", 8: "PKV_ERR_REQUEST_TOO_LARGE",
    9: "PKV_ERR_TIMEOUT",
}
OK, ERR_INVALID_ARGUMENT, ERR_DEVICE_INDEX, ERR_POOL_EXHAUSTED = 0, 1, 6, 7
ERR_REQUEST_TOO_LARGE, ERR_TIMEOUT = 8, 9


class PkvError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        msg = f"{where}: {STATUS.get(status, status)}"
        super().__init__(msg + (f" ({detail})" if detail else ""))


_p, _i, _f, _d, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_double, ctypes.c_size_t
_ip = ctypes.POINTER(ctypes.c_int)


class DecodeOpts(ctypes.Structure):
    _fields_ = [("compute", _i), ("min_units_per_warp", _i), ("ctas_per_sm", _i), ("stages", _i),
                ("warps_per_cta", _i), ("combine", _i), ("schedule", _i), ("early_kv", _i),
                ("wait_limit_ns", ctypes.c_longlong), ("expire_first_wait", _i)]


_SIGS = {
    "pkv_status_string": (ctypes.c_char_p, [_i]),
    "pkv_version": (_i, []),
    "pkv_last_error": (ctypes.c_char_p, []),
    "pkv_rope_inv_freq_plain": (_i, [_p, _d]),
    "pkv_rope_inv_freq_llama3": (_i, [_p, _d, _d, _d, _d, _i]),
    "pkv_rope_table_fill": (_i, [_p, _p, _i, _p]),
    "kv_append_rope": (_i, [_p, _p, _p, _p, _i, _p, _i, _i, _i, _p, _i, _p, _p, _i, _p, _p, _p, _p]),
    "paged_gqa_decode_workspace_bytes": (_sz, [_i]),
    "paged_gqa_prefill": (_i, [_p, _i, _p, _p, _i, _p, _i, _i, _p, _i, _i, _p, _f, _p, _p]),
    "paged_gqa_prefill_ex": (_i, [_p, _i, _p, _p, _i, _p, _i, _i, _p, _i, _i, _p, _f, _p, _p, _i]),
    "pkv_argmax_f32": (_i, [_p, _i, _i, ctypes.c_longlong, _p, _p]),
    "paged_gqa_decode": (_i, [_p, _p, _i, _p, _i, _i, _p, _i, _i, _p, _f, _p, _sz, _p, _p]),
    "paged_gqa_decode_ex": (_i, [_p, _p, _i, _p, _i, _i, _p, _i, _i, _p, _f, _p, _sz, _p, _p,
                                 ctypes.POINTER(DecodeOpts)]),
    "paged_gqa_decode_append": (_i, [_p, _p, _p, _p, _p, _i, _p, _i, _p, _i, _i, _p, _i, _i, _p, _p,
                                     _f, _p, _sz, _p, _p, ctypes.POINTER(DecodeOpts)]),
    "paged_gqa_decode_noalloc": (_i, [_p, _p, _i, _p, _i, _i, _p, _i, _i, _p, _f, _p, _p]),
    "kv_append_rope_int8": (_i, [_p, _p, _p, _p, _i, _p, _i, _i, _i, _p, _i, _p, _p, _i, _p, _p, _p,
                                 _p]),
    "kv_append_rope_layers": (_i, [_p, _p, _i, _i, _p, _sz, _p, _p, _i, _p, ctypes.c_longlong, _i,
                                   _i, _i, _p, _i, _i, _p, _p, _i, _p, _p]),
    "paged_gqa_decode_int8": (_i, [_p, _p, _i, _p, _i, _i, _p, _i, _i, _p, _f, _p, _sz, _p, _p]),
    "paged_gqa_decode_int8_ex": (_i, [_p, _p, _i, _p, _i, _i, _p, _i, _i, _p, _f, _p, _sz, _p, _p,
                                      ctypes.POINTER(DecodeOpts)]),
    "paged_gqa_decode_append_int8": (_i, [_p, _p, _p, _p, _p, _i, _p, _i, _p, _i, _i, _p, _i, _i, _p,
                                          _p, _f, _p, _sz, _p, _p, ctypes.POINTER(DecodeOpts)]),
    "paged_gqa_decode_append_layers": (_i, [_p, _p, _p, _p, _p, _i, _i, _p, _p, _i, _p, _i, _i, _p,
                                            ctypes.c_longlong, _i, _i, _p, _i, _f, _p, _sz, _p, _p,
                                            _i, _p, _p, _sz]),
    "pkv_read_device_error": (_i, [_p, _p, _i, _ip]),
    "pkv_credit_pages": (_i, [_i, _i, _i]),
    "pkv_sched_create": (_p, [_i, _i, _i, _i]),
    "pkv_sched_set_mode": (_i, [_p, _i]),
    "pkv_sched_destroy": (None, [_p]),
    "pkv_sched_submit": (_i, [_p, _i, _i, _ip]),
    "pkv_sched_admit": (_i, [_p, _p, _i, _ip]),
    "pkv_sched_grow": (_i, [_p, _i, _i]),
    "pkv_sched_finish": (_i, [_p, _i]),
    "pkv_sched_block_table": (_i, [_p, _i, _i, _p, _ip]),
    "pkv_sched_stats": (_i, [_p, _ip, _ip, _ip, _ip]),
    "pkv_sched_event_count": (_i, [_p]),
    "pkv_sched_event": (_i, [_p, _i, _ip, _ip, _ip, _ip]),
    "pkv_sched_begin_step": (_i, [_p, _p, _p, _i, _ip]),
    "pkv_sched_step_bytes": (_sz, [_p, _i, _i]),
    "pkv_sched_pack_step": (_i, [_p, _p, _i, _i, _p, _sz]),
}

_LIB = None


def _L():
    """The loaded libpkv.so; raises if it has not been built (no fallback exists)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libpkv.so not found at {LIB_PATH}; build it with "
                               "`python -m paged_kv_gqa_append_gb300.build` (nvcc, sm_103a)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def __getattr__(name):
    if name == "lib":
        return _L()
    raise AttributeError(name)


def _check(status: int, where: str):
    if status != OK:
        detail = _L().pkv_last_error().decode() if status == 5 else ""
        raise PkvError(status, where, detail)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, name, dtype, device=None, shape_tail=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if shape_tail is not None and tuple(t.shape[-len(shape_tail):]) != tuple(shape_tail):
        raise ValueError(f"{name} must end in shape {shape_tail}, got {tuple(t.shape)}")


def status_string(status: int) -> str:
    return _L().pkv_status_string(status).decode()


# --------------------------------------------------------------- RoPE set-up --

def pkv_rope_inv_freq_plain(theta: float = 500000.0) -> np.ndarray:
    out = np.zeros(ROPE_PAIRS, np.float64)
    _check(_L().pkv_rope_inv_freq_plain(out.ctypes.data, theta), "pkv_rope_inv_freq_plain")
    return out


def pkv_rope_inv_freq_llama3(theta=500000.0, factor=32.0, low_freq_factor=1.0,
                             high_freq_factor=4.0, original_max_pos=8192) -> np.ndarray:
    out = np.zeros(ROPE_PAIRS, np.float64)
    _check(_L().pkv_rope_inv_freq_llama3(out.ctypes.data, theta, factor, low_freq_factor,
                                        high_freq_factor, original_max_pos),
           "pkv_rope_inv_freq_llama3")
    return out


def pkv_rope_table_fill(inv_freq, max_pos: int):
    """Host fp32 cos/sin tables [max_pos][32] (numpy)."""
    f = np.ascontiguousarray(inv_freq, dtype=np.float64)
    if f.shape != (ROPE_PAIRS,):
        raise ValueError("inv_freq must have 32 entries")
    cos = np.empty((max_pos, ROPE_PAIRS), np.float32)
    sin = np.empty_like(cos)
    _check(_L().pkv_rope_table_fill(cos.ctypes.data, sin.ctypes.data, max_pos, f.ctypes.data),
           "pkv_rope_table_fill")
    return cos, sin


def rope_tables_device(device, max_pos: int = 2048, inv_freq=None):
    """cos/sin tables on `device` (Llama-3.2 frequencies by default)."""
    if inv_freq is None:
        inv_freq = pkv_rope_inv_freq_llama3()
    cos, sin = pkv_rope_table_fill(inv_freq, max_pos)
    return torch.from_numpy(cos).to(device), torch.from_numpy(sin).to(device)


# ------------------------------------------------------------------- append --

def kv_append_rope(k, v, positions, block_tables, kv_pool, rope_cos, rope_sin,
                   token_seq=None, q_in=None, q_out=None, d_err=None, max_blocks=None,
                   stream=None):
    """Rotate K (and optionally q) at `positions` and write K/V into pool pages."""
    dev = kv_pool.device
    _need(kv_pool, "kv_pool", torch.bfloat16, dev, (2, NUM_KV_HEADS, PAGE_TOKENS, HEAD_DIM))
    _need(k, "k", torch.bfloat16, dev, (NUM_KV_HEADS, HEAD_DIM))
    _need(v, "v", torch.bfloat16, dev, (NUM_KV_HEADS, HEAD_DIM))
    T = k.numel() // (NUM_KV_HEADS * HEAD_DIM)
    if v.numel() != k.numel():
        raise ValueError("k and v must have the same shape")
    _need(positions, "positions", torch.int32, dev)
    if positions.numel() != T:
        raise ValueError("positions must have one entry per token")
    if token_seq is not None:
        _need(token_seq, "token_seq", torch.int32, dev)
        if token_seq.numel() != T:
            raise ValueError("token_seq must have one entry per token")
    _need(block_tables, "block_tables", torch.int32, dev)
    if block_tables.dim() != 2:
        raise ValueError("block_tables must be [num_seqs, row_stride]")
    _need(rope_cos, "rope_cos", torch.float32, dev, (ROPE_PAIRS,))
    _need(rope_sin, "rope_sin", torch.float32, dev, (ROPE_PAIRS,))
    if (q_in is None) != (q_out is None):
        raise ValueError("q_in and q_out go together")
    if q_in is not None:
        _need(q_in, "q_in", torch.bfloat16, dev, (NUM_Q_HEADS, HEAD_DIM))
        _need(q_out, "q_out", torch.bfloat16, dev, (NUM_Q_HEADS, HEAD_DIM))
        if q_in.numel() != T * NUM_Q_HEADS * HEAD_DIM or q_out.numel() != q_in.numel():
            raise ValueError("q_in/q_out must be [T, 32, 64]")
    if d_err is not None:
        _need(d_err, "d_err", torch.int32, dev)
    S, stride = block_tables.shape
    mb = stride if max_blocks is None else max_blocks
    st = _L().kv_append_rope(_ptr(k), _ptr(v), _ptr(positions), _ptr(token_seq), T,
                            _ptr(block_tables), S, stride, mb, _ptr(kv_pool), kv_pool.shape[0],
                            _ptr(rope_cos), _ptr(rope_sin), rope_cos.shape[0],
                            _ptr(q_in), _ptr(q_out), _ptr(d_err), _stream(stream))
    _check(st, "kv_append_rope")


# ------------------------------------------------------------------- decode --

def paged_gqa_decode_workspace_bytes(num_seqs: int) -> int:
    return int(_L().paged_gqa_decode_workspace_bytes(num_seqs))


def alloc_workspace(num_seqs: int, device) -> torch.Tensor:
    """Caller-owned workspace for paged_gqa_decode, zero-filled as the call requires."""
    with torch.cuda.device(device):
        n = paged_gqa_decode_workspace_bytes(num_seqs)
    if n <= 0:
        raise PkvError(5, "paged_gqa_decode_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def paged_gqa_decode(q, kv_pool, block_tables, seq_lens, out, scale, workspace=None,
                     max_seq_len=None, d_err=None, max_blocks=None, compute=None,
                     min_units_per_warp=0, ctas_per_sm=0, stages=0, warps_per_cta=0,
                     combine=0, schedule=None, early_kv=0, stream=None, wait_limit_ns=0,
                     expire_first_wait=0):
    """out[s, h] = softmax(scale * q[s, h] . K) V over sequence s's own pages.

    early_kv=1 promises that the kernel enqueued just before this call on the
    stream writes neither block_tables, seq_lens nor the pages read here; the
    call then starts on them while that kernel finishes.  schedule: None or
    SCHEDULE_AUTO (by work per SM), SCHEDULE_STATIC or SCHEDULE_DYNAMIC.
    wait_limit_ns and expire_first_wait: the bounded-wait limit and its test
    (pkv_decode_opts).
    """
    dev = kv_pool.device
    _need(kv_pool, "kv_pool", torch.bfloat16, dev, (2, NUM_KV_HEADS, PAGE_TOKENS, HEAD_DIM))
    _need(q, "q", torch.bfloat16, dev, (NUM_Q_HEADS, HEAD_DIM))
    _need(out, "out", torch.bfloat16, dev, (NUM_Q_HEADS, HEAD_DIM))
    S = q.numel() // (NUM_Q_HEADS * HEAD_DIM)
    if out.numel() != q.numel():
        raise ValueError("out must match q")
    _need(block_tables, "block_tables", torch.int32, dev)
    if block_tables.dim() != 2 or block_tables.shape[0] < S:
        raise ValueError("block_tables must be [>= num_seqs, row_stride]")
    _need(seq_lens, "seq_lens", torch.int32, dev)
    if seq_lens.numel() != S:
        raise ValueError("seq_lens must have num_seqs entries")
    stride = block_tables.shape[1]
    mb = stride if max_blocks is None else max_blocks
    if max_seq_len is None:
        max_seq_len = PAGE_TOKENS * mb
    if workspace is None:
        workspace = alloc_workspace(S, dev)
    _need(workspace, "workspace", torch.uint8, dev)
    if d_err is not None:
        _need(d_err, "d_err", torch.int32, dev)
    args = (_ptr(q), _ptr(kv_pool), kv_pool.shape[0], _ptr(block_tables), stride, mb,
            _ptr(seq_lens), S, int(max_seq_len), _ptr(out), float(scale), _ptr(workspace),
            workspace.numel(), _ptr(d_err), _stream(stream))
    if compute is None and not (min_units_per_warp or ctas_per_sm or stages or warps_per_cta
                                or combine or schedule is not None or early_kv
                                or wait_limit_ns or expire_first_wait):
        st = _L().paged_gqa_decode(*args)
    else:
        opts = DecodeOpts(COMPUTE_TENSOR if compute is None else compute,
                          min_units_per_warp, ctas_per_sm, stages, warps_per_cta, combine,
                          SCHEDULE_AUTO if schedule is None else schedule, early_kv,
                          wait_limit_ns, expire_first_wait)
        st = _L().paged_gqa_decode_ex(*args, ctypes.byref(opts))
    _check(st, "paged_gqa_decode")


# --------------------------------------------------------------- INT8 pages --

I8_BLOCK_BYTES = 2 * PAGE_TOKENS * HEAD_DIM + 2 * PAGE_TOKENS * 4   # 2176 per (page, KV head)


def new_int8_pool(num_pages: int, device) -> torch.Tensor:
    """An empty INT8 pool, uint8 [num_pages, 8, 2176]: every code 0 (stored as
    the byte 0x80) and every scale 0.  The block format is in pkv.h."""
    pool = torch.zeros((num_pages, NUM_KV_HEADS, I8_BLOCK_BYTES), dtype=torch.uint8, device=device)
    pool[:, :, :2 * 16 * 64] = 0x80
    return pool


def _need_i8_pool(kv_pool, dev):
    _need(kv_pool, "kv_pool", torch.uint8, dev, (NUM_KV_HEADS, I8_BLOCK_BYTES))
    if kv_pool.dim() != 3:
        raise ValueError("the INT8 pool must be [num_pages, 8, 2176] uint8")


def kv_append_rope_layers(k, v, positions, block_tables, kv_pool, rope_cos, rope_sin,
                          token_seq=None, stage=None, d_err=None, max_blocks=None, stream=None):
    """The same T tokens appended into every layer in one native call (a new
    request's prompt).  k, v: sequences of L tensors [T, 8, 64] bf16, all on
    the pool's device, or all in host memory (pinned for an asynchronous
    copy; each layer's rows then pass through `stage`, a device uint8 tensor
    of at least 2 * T * 1024 bytes).  block_tables: [L, num_seqs, >= max_blocks]
    int32 with unit stride in its last dimension (any layer and row strides,
    e.g. the one-row view of a request in a larger table).  kv_pool: a bf16
    pool or an INT8 pool (new_int8_pool).  No q rotation."""
    dev = kv_pool.device
    int8 = kv_pool.dtype == torch.uint8
    if int8:
        _need_i8_pool(kv_pool, dev)
    else:
        _need(kv_pool, "kv_pool", torch.bfloat16, dev, (2, NUM_KV_HEADS, PAGE_TOKENS, HEAD_DIM))
    L = len(k)
    if len(v) != L:
        raise ValueError("k and v must hold one tensor per layer each")
    if L == 0:
        return
    src_host = k[0].device.type == "cpu"
    where = torch.device("cpu") if src_host else dev
    T = k[0].numel() // (NUM_KV_HEADS * HEAD_DIM)
    for i, t in enumerate(list(k) + list(v)):
        _need(t, f"{'kv'[i // L]}[{i % L}]", torch.bfloat16, where, (NUM_KV_HEADS, HEAD_DIM))
        if t.numel() != T * NUM_KV_HEADS * HEAD_DIM:
            raise ValueError("every layer's k and v must be [T, 8, 64]")
    _need(positions, "positions", torch.int32, dev)
    if positions.numel() != T:
        raise ValueError("positions must have one entry per token")
    if token_seq is not None:
        _need(token_seq, "token_seq", torch.int32, dev)
        if token_seq.numel() != T:
            raise ValueError("token_seq must have one entry per token")
    if (not isinstance(block_tables, torch.Tensor) or block_tables.dtype != torch.int32 or
            block_tables.device != dev or block_tables.dim() != 3 or block_tables.stride(2) != 1):
        raise ValueError("block_tables must be an int32 [L, num_seqs, row] tensor on the pool's "
                         "device with unit stride in its last dimension")
    if block_tables.shape[0] < L:
        raise ValueError("block_tables must hold one table per layer")
    _need(rope_cos, "rope_cos", torch.float32, dev, (ROPE_PAIRS,))
    _need(rope_sin, "rope_sin", torch.float32, dev, (ROPE_PAIRS,))
    if src_host:
        _need(stage, "stage", torch.uint8, dev)
        if stage.numel() < 2 * T * NUM_KV_HEADS * HEAD_DIM * 2:
            raise ValueError("stage must hold 2 * T * 1024 bytes")
    if d_err is not None:
        _need(d_err, "d_err", torch.int32, dev)
    S, mb0 = block_tables.shape[1], block_tables.shape[2]
    ks = (ctypes.c_void_p * L)(*[t.data_ptr() for t in k])
    vs = (ctypes.c_void_p * L)(*[t.data_ptr() for t in v])
    st = _L().kv_append_rope_layers(
        ks, vs, L, int(src_host), _ptr(stage) if src_host else None,
        stage.numel() if src_host else 0, _ptr(positions), _ptr(token_seq), T,
        _ptr(block_tables), block_tables.stride(0), S, block_tables.stride(1),
        mb0 if max_blocks is None else max_blocks, _ptr(kv_pool), kv_pool.shape[0], int(int8),
        _ptr(rope_cos), _ptr(rope_sin), rope_cos.shape[0], _ptr(d_err), _stream(stream))
    _check(st, "kv_append_rope_layers")


def kv_append_rope_int8(k, v, positions, block_tables, kv_pool, rope_cos, rope_sin,
                        token_seq=None, q_in=None, q_out=None, d_err=None, max_blocks=None,
                        stream=None):
    """kv_append_rope into INT8 pages: each (token, head) row of the rotated K
    and of V is stored as 64 int8 codes and one fp32 scale."""
    dev = kv_pool.device
    _need_i8_pool(kv_pool, dev)
    _need(k, "k", torch.bfloat16, dev, (NUM_KV_HEADS, HEAD_DIM))
    _need(v, "v", torch.bfloat16, dev, (NUM_KV_HEADS, HEAD_DIM))
    T = k.numel() // (NUM_KV_HEADS * HEAD_DIM)
    if v.numel() != k.numel():
        raise ValueError("k and v must have the same shape")
    _need(positions, "positions", torch.int32, dev)
    if positions.numel() != T:
        raise ValueError("positions must have one entry per token")
    if token_seq is not None:
        _need(token_seq, "token_seq", torch.int32, dev)
        if token_seq.numel() != T:
            raise ValueError("token_seq must have one entry per token")
    _need(block_tables, "block_tables", torch.int32, dev)
    if block_tables.dim() != 2:
        raise ValueError("block_tables must be [num_seqs, row_stride]")
    _need(rope_cos, "rope_cos", torch.float32, dev, (ROPE_PAIRS,))
    _need(rope_sin, "rope_sin", torch.float32, dev, (ROPE_PAIRS,))
    if (q_in is None) != (q_out is None):
        raise ValueError("q_in and q_out go together")
    if q_in is not None:
        _need(q_in, "q_in", torch.bfloat16, dev, (NUM_Q_HEADS, HEAD_DIM))
        _need(q_out, "q_out", torch.bfloat16, dev, (NUM_Q_HEADS, HEAD_DIM))
        if q_in.numel() != T * NUM_Q_HEADS * HEAD_DIM or q_out.numel() != q_in.numel():
            raise ValueError("q_in/q_out must be [T, 32, 64]")
    if d_err is not None:
        _need(d_err, "d_err", torch.int32, dev)
    S, stride = block_tables.shape
    mb = stride if max_blocks is None else max_blocks
    st = _L().kv_append_rope_int8(_ptr(k), _ptr(v), _ptr(positions), _ptr(token_seq), T,
                                 _ptr(block_tables), S, stride, mb, _ptr(kv_pool), kv_pool.shape[0],
                                 _ptr(rope_cos), _ptr(rope_sin), rope_cos.shape[0], _ptr(q_in),
                                 _ptr(q_out), _ptr(d_err), _stream(stream))
    _check(st, "kv_append_rope_int8")


def paged_gqa_decode_int8(q, kv_pool, block_tables, seq_lens, out, scale, workspace=None,
                          max_seq_len=None, d_err=None, max_blocks=None, min_units_per_warp=0,
                          ctas_per_sm=0, stages=0, warps_per_cta=0, early_kv=0, stream=None):
    """paged_gqa_decode over INT8 pages (early_kv as for paged_gqa_decode: the
    lengths, tables and first pages are read before the previous kernel on the
    stream has finished, which must not write them)."""
    dev = kv_pool.device
    _need_i8_pool(kv_pool, dev)
    _need(q, "q", torch.bfloat16, dev, (NUM_Q_HEADS, HEAD_DIM))
    _need(out, "out", torch.bfloat16, dev, (NUM_Q_HEADS, HEAD_DIM))
    S = q.numel() // (NUM_Q_HEADS * HEAD_DIM)
    if out.numel() != q.numel():
        raise ValueError("out must match q")
    _need(block_tables, "block_tables", torch.int32, dev)
    if block_tables.dim() != 2 or block_tables.shape[0] < S:
        raise ValueError("block_tables must be [>= num_seqs, row_stride]")
    _need(seq_lens, "seq_lens", torch.int32, dev)
    if seq_lens.numel() != S:
        raise ValueError("seq_lens must have num_seqs entries")
    stride = block_tables.shape[1]
    mb = stride if max_blocks is None else max_blocks
    if max_seq_len is None:
        max_seq_len = PAGE_TOKENS * mb
    if workspace is None:
        workspace = alloc_workspace(S, dev)
    _need(workspace, "workspace", torch.uint8, dev)
    if d_err is not None:
        _need(d_err, "d_err", torch.int32, dev)
    args = (_ptr(q), _ptr(kv_pool), kv_pool.shape[0], _ptr(block_tables), stride, mb,
            _ptr(seq_lens), S, int(max_seq_len), _ptr(out), float(scale), _ptr(workspace),
            workspace.numel(), _ptr(d_err), _stream(stream))
    if not (min_units_per_warp or ctas_per_sm or stages or warps_per_cta or early_kv):
        st = _L().paged_gqa_decode_int8(*args)
    else:
        opts = DecodeOpts(COMPUTE_TENSOR, min_units_per_warp, ctas_per_sm, stages, warps_per_cta,
                          0, SCHEDULE_AUTO, int(bool(early_kv)))
        st = _L().paged_gqa_decode_int8_ex(*args, ctypes.byref(opts))
    _check(st, "paged_gqa_decode_int8")


def paged_gqa_decode_append_int8(q, k_new, v_new, kv_pool, block_tables, seq_lens, out, rope_cos,
                                 rope_sin, scale, q_out=None, workspace=None, max_seq_len=None,
                                 d_err=None, max_blocks=None, min_units_per_warp=0, early_kv=0,
                                 stream=None):
    """paged_gqa_decode_append on INT8 pages: sequence s's new token (k_new[s],
    v_new[s]) is quantised into its page at seq_lens[s] - 1 and q rotated
    there, then attention over seq_lens[s] tokens -- one kernel."""
    dev = kv_pool.device
    _need_i8_pool(kv_pool, dev)
    _need(q, "q", torch.bfloat16, dev, (NUM_Q_HEADS, HEAD_DIM))
    _need(out, "out", torch.bfloat16, dev, (NUM_Q_HEADS, HEAD_DIM))
    S = q.numel() // (NUM_Q_HEADS * HEAD_DIM)
    if out.numel() != q.numel():
        raise ValueError("out must match q")
    _need(k_new, "k_new", torch.bfloat16, dev, (NUM_KV_HEADS, HEAD_DIM))
    _need(v_new, "v_new", torch.bfloat16, dev, (NUM_KV_HEADS, HEAD_DIM))
    if k_new.numel() != S * NUM_KV_HEADS * HEAD_DIM or v_new.numel() != k_new.numel():
        raise ValueError("k_new/v_new must be [num_seqs, 8, 64]")
    if q_out is not None:
        _need(q_out, "q_out", torch.bfloat16, dev, (NUM_Q_HEADS, HEAD_DIM))
        if q_out.numel() != q.numel():
            raise ValueError("q_out must match q")
    _need(block_tables, "block_tables", torch.int32, dev)
    if block_tables.dim() != 2 or block_tables.shape[0] < S:
        raise ValueError("block_tables must be [>= num_seqs, row_stride]")
    _need(seq_lens, "seq_lens", torch.int32, dev)
    if seq_lens.numel() != S:
        raise ValueError("seq_lens must have num_seqs entries")
    _need(rope_cos, "rope_cos", torch.float32, dev, (ROPE_PAIRS,))
    _need(rope_sin, "rope_sin", torch.float32, dev, (ROPE_PAIRS,))
    stride = block_tables.shape[1]
    mb = stride if max_blocks is None else max_blocks
    if max_seq_len is None:
        max_seq_len = PAGE_TOKENS * mb
    if workspace is None:
        workspace = alloc_workspace(S, dev)
    _need(workspace, "workspace", torch.uint8, dev)
    if d_err is not None:
        _need(d_err, "d_err", torch.int32, dev)
    opts = DecodeOpts(COMPUTE_TENSOR, min_units_per_warp, 0, 0, 0, 0, SCHEDULE_AUTO, early_kv)
    st = _L().paged_gqa_decode_append_int8(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(rope_cos), _ptr(rope_sin), rope_cos.shape[0],
        _ptr(kv_pool), kv_pool.shape[0], _ptr(block_tables), stride, mb, _ptr(seq_lens), S,
        int(max_seq_len), _ptr(q_out), _ptr(out), float(scale), _ptr(workspace), workspace.numel(),
        _ptr(d_err), _stream(stream), ctypes.byref(opts))
    _check(st, "paged_gqa_decode_append_int8")


def paged_gqa_decode_append(q, k_new, v_new, kv_pool, block_tables, seq_lens, out, rope_cos,
                            rope_sin, scale, q_out=None, workspace=None, max_seq_len=None,
                            d_err=None, max_blocks=None, warps_per_cta=0, min_units_per_warp=0,
                            ctas_per_sm=0, schedule=None, early_kv=0, stream=None):
    """One decode step: append each sequence's new token at seq_lens-1, then attend.

    early_kv as for paged_gqa_decode (the pages meant are the ones this call
    reads and appends to).
    """
    dev = kv_pool.device
    _need(kv_pool, "kv_pool", torch.bfloat16, dev, (2, NUM_KV_HEADS, PAGE_TOKENS, HEAD_DIM))
    _need(q, "q", torch.bfloat16, dev, (NUM_Q_HEADS, HEAD_DIM))
    _need(out, "out", torch.bfloat16, dev, (NUM_Q_HEADS, HEAD_DIM))
    S = q.numel() // (NUM_Q_HEADS * HEAD_DIM)
    if out.numel() != q.numel():
        raise ValueError("out must match q")
    for t, name in ((k_new, "k_new"), (v_new, "v_new")):
        _need(t, name, torch.bfloat16, dev, (NUM_KV_HEADS, HEAD_DIM))
        if t.numel() != S * NUM_KV_HEADS * HEAD_DIM:
            raise ValueError(f"{name} must be [num_seqs, 8, 64]")
    if q_out is not None:
        _need(q_out, "q_out", torch.bfloat16, dev, (NUM_Q_HEADS, HEAD_DIM))
        if q_out.numel() != q.numel():
            raise ValueError("q_out must match q")
    _need(rope_cos, "rope_cos", torch.float32, dev, (ROPE_PAIRS,))
    _need(rope_sin, "rope_sin", torch.float32, dev, (ROPE_PAIRS,))
    _need(block_tables, "block_tables", torch.int32, dev)
    if block_tables.dim() != 2 or block_tables.shape[0] < S:
        raise ValueError("block_tables must be [>= num_seqs, row_stride]")
    _need(seq_lens, "seq_lens", torch.int32, dev)
    if seq_lens.numel() != S:
        raise ValueError("seq_lens must have num_seqs entries")
    stride = block_tables.shape[1]
    mb = stride if max_blocks is None else max_blocks
    if max_seq_len is None:
        max_seq_len = PAGE_TOKENS * mb
    if workspace is None:
        workspace = alloc_workspace(S, dev)
    _need(workspace, "workspace", torch.uint8, dev)
    if d_err is not None:
        _need(d_err, "d_err", torch.int32, dev)
    opts = DecodeOpts(COMPUTE_TENSOR, min_units_per_warp, ctas_per_sm, 0, warps_per_cta, 0,
                      SCHEDULE_AUTO if schedule is None else schedule, early_kv)
    st = _L().paged_gqa_decode_append(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(rope_cos), _ptr(rope_sin), rope_cos.shape[0],
        _ptr(kv_pool), kv_pool.shape[0], _ptr(block_tables), stride, mb, _ptr(seq_lens), S,
        int(max_seq_len), _ptr(q_out), _ptr(out), float(scale), _ptr(workspace),
        workspace.numel(), _ptr(d_err), _stream(stream), ctypes.byref(opts))
    _check(st, "paged_gqa_decode_append")


def paged_gqa_decode_append_layers(q, k_new, v_new, kv_pool, block_tables, seq_lens, out,
                                   rope_cos, rope_sin, scale, workspace, max_seq_len=None,
                                   d_err=None, stream=None, q_out=None, early_kv=1,
                                   host_stage=None, dev_stage=None, check=True):
    """A whole decode step: for every layer l, the fused append + decode of
    q[l], k_new[l], v_new[l] over block_tables[l] into out[l] on a bf16 pool
    (paged_gqa_decode_append) or an INT8 pool (paged_gqa_decode_append_int8),
    in layer order on one stream -- one call of the C function of the same
    name, which makes those per-layer calls.

    q, out (and q_out): [L, S, 32, 64] bf16; k_new, v_new: [L, S, 8, 64] bf16;
    block_tables: [L, S', row_stride] int32 with S' >= S; seq_lens: [S] int32,
    shared by the layers.  early_kv=1 lets layers >= 1 read their tables and
    stage their first pages while the previous layer's kernel finishes (the
    layers' pages must be disjoint).  host_stage (pinned uint8 host tensor) and
    dev_stage (uint8 device tensor of at least its size): one copy of the
    first into the second runs on the stream before the launches, e.g. the
    block of pkv_sched_pack_step that block_tables / seq_lens are views of.
    check=False skips the tensor checks below (the C call still checks sizes,
    pointers and alignment): for a caller that built the tensors itself and
    checked their shapes once, as ContinuousBatcher does every step.
    """
    dev = kv_pool.device
    int8 = kv_pool.dtype == torch.uint8
    if check:
        _check_layers_args(q, k_new, v_new, kv_pool, block_tables, seq_lens, out, rope_cos,
                           rope_sin, workspace, d_err, q_out, host_stage, dev_stage, int8, dev)
    L, S = q.shape[0], q.shape[1]
    if L == 0:
        return
    stage = 0 if host_stage is None else host_stage.numel()
    stride = block_tables.shape[2]
    if max_seq_len is None:
        max_seq_len = PAGE_TOKENS * stride
    st = _L().paged_gqa_decode_append_layers(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(q_out), _ptr(out), L, S, _ptr(rope_cos),
        _ptr(rope_sin), rope_cos.shape[0], _ptr(kv_pool), kv_pool.shape[0], int(int8),
        _ptr(block_tables), block_tables.shape[1] * stride, stride, stride, _ptr(seq_lens),
        int(max_seq_len), float(scale), _ptr(workspace), workspace.numel(), _ptr(d_err),
        _stream(stream), int(early_kv), _ptr(host_stage), _ptr(dev_stage), stage)
    _check(st, "paged_gqa_decode_append_layers")


def _check_layers_args(q, k_new, v_new, kv_pool, block_tables, seq_lens, out, rope_cos, rope_sin,
                       workspace, d_err, q_out, host_stage, dev_stage, int8, dev):
    if int8:
        _need_i8_pool(kv_pool, dev)
    else:
        _need(kv_pool, "kv_pool", torch.bfloat16, dev, (2, NUM_KV_HEADS, PAGE_TOKENS, HEAD_DIM))
    for t, name, heads in ((q, "q", NUM_Q_HEADS), (out, "out", NUM_Q_HEADS),
                           (k_new, "k_new", NUM_KV_HEADS), (v_new, "v_new", NUM_KV_HEADS)):
        _need(t, name, torch.bfloat16, dev, (heads, HEAD_DIM))
        if t.dim() != 4:
            raise ValueError(f"{name} must be [layers, num_seqs, {heads}, {HEAD_DIM}]")
    L, S = q.shape[0], q.shape[1]
    if out.shape != q.shape or k_new.shape[:2] != (L, S) or v_new.shape != k_new.shape:
        raise ValueError("q/out [L, S, 32, 64] and k_new/v_new [L, S, 8, 64] must agree")
    if q_out is not None:
        _need(q_out, "q_out", torch.bfloat16, dev, (NUM_Q_HEADS, HEAD_DIM))
        if q_out.shape != q.shape:
            raise ValueError("q_out must match q")
    if L == 0:
        return
    _need(block_tables, "block_tables", torch.int32, dev)
    if block_tables.dim() != 3 or block_tables.shape[0] != L or block_tables.shape[1] < S:
        raise ValueError("block_tables must be [layers, >= num_seqs, row_stride]")
    _need(seq_lens, "seq_lens", torch.int32, dev)
    if seq_lens.numel() != S:
        raise ValueError("seq_lens must have num_seqs entries")
    _need(rope_cos, "rope_cos", torch.float32, dev, (ROPE_PAIRS,))
    _need(rope_sin, "rope_sin", torch.float32, dev, (ROPE_PAIRS,))
    _need(workspace, "workspace", torch.uint8, dev)
    if d_err is not None:
        _need(d_err, "d_err", torch.int32, dev)
    if (host_stage is None) != (dev_stage is None):
        raise ValueError("host_stage and dev_stage go together")
    if host_stage is not None:
        if host_stage.dtype != torch.uint8 or not host_stage.is_contiguous():
            raise TypeError("host_stage must be a contiguous uint8 host tensor")
        _need(dev_stage, "dev_stage", torch.uint8, dev)
        if dev_stage.numel() < host_stage.numel():
            raise ValueError("dev_stage is smaller than host_stage")


PREFILL_MMA_SYNC = 2  # comparison arm of paged_gqa_prefill (legacy bf16 mma.sync)


def paged_gqa_prefill(q, cu_q, kv_pool, block_tables, seq_lens, out, scale, max_q_len=None,
                      d_err=None, max_blocks=None, compute=None, stream=None):
    """Causal attention of each sequence's last q_len tokens over its own pages.

    q, out: [T, 32, 64] bf16 (q rotated); cu_q: [S + 1] int32 row offsets on
    the device; seq_lens: [S] int32 tokens held (the queries are the last
    cu_q[s+1] - cu_q[s] of them).  max_q_len: host bound of every q_len
    (default T).  compute: None / COMPUTE_TENSOR (tcgen05, tensor memory) or
    PREFILL_MMA_SYNC.
    """
    dev = kv_pool.device
    _need(kv_pool, "kv_pool", torch.bfloat16, dev, (2, NUM_KV_HEADS, PAGE_TOKENS, HEAD_DIM))
    _need(q, "q", torch.bfloat16, dev, (NUM_Q_HEADS, HEAD_DIM))
    _need(out, "out", torch.bfloat16, dev, (NUM_Q_HEADS, HEAD_DIM))
    T = q.numel() // (NUM_Q_HEADS * HEAD_DIM)
    if out.numel() != q.numel():
        raise ValueError("out must match q")
    _need(cu_q, "cu_q", torch.int32, dev)
    _need(seq_lens, "seq_lens", torch.int32, dev)
    S = seq_lens.numel()
    if cu_q.numel() != S + 1:
        raise ValueError("cu_q must have num_seqs + 1 entries")
    _need(block_tables, "block_tables", torch.int32, dev)
    if block_tables.dim() != 2 or block_tables.shape[0] < S:
        raise ValueError("block_tables must be [>= num_seqs, row_stride]")
    stride = block_tables.shape[1]
    mb = stride if max_blocks is None else max_blocks
    if d_err is not None:
        _need(d_err, "d_err", torch.int32, dev)
    st = _L().paged_gqa_prefill_ex(_ptr(q), T, _ptr(cu_q), _ptr(kv_pool), kv_pool.shape[0],
                                   _ptr(block_tables), stride, mb, _ptr(seq_lens), S,
                                   int(T if max_q_len is None else max_q_len), _ptr(out),
                                   float(scale), _ptr(d_err), _stream(stream),
                                   COMPUTE_TENSOR if compute is None else int(compute))
    _check(st, "paged_gqa_prefill")


def argmax_rows(logits, out=None, stream=None):
    """Next-token ids: per row of FP32 logits [rows, vocab] (row stride may
    exceed vocab), the first index of the largest non-NaN value."""
    if logits.dtype != torch.float32 or not logits.is_cuda or logits.dim() != 2:
        raise ValueError("logits must be a 2-D float32 CUDA tensor")
    if logits.stride(1) != 1:
        raise ValueError("logits rows must be contiguous")
    rows, vocab = logits.shape
    if out is None:
        out = torch.empty(rows, dtype=torch.int32, device=logits.device)
    _need(out, "out", torch.int32, logits.device)
    _check(_L().pkv_argmax_f32(_ptr(logits), rows, vocab, logits.stride(0), _ptr(out),
                               _stream(stream)), "pkv_argmax_f32")
    return out


def pkv_read_device_error(d_err, clear: bool = True, stream=None) -> int:
    """Synchronise the stream and return the device error word (optionally reset it)."""
    code = ctypes.c_int(0)
    _check(_L().pkv_read_device_error(_ptr(d_err), _stream(stream), int(clear), ctypes.byref(code)),
           "pkv_read_device_error")
    return code.value


# ---------------------------------------------------------------- scheduler --

def pkv_credit_pages(prompt_tokens: int, allowed_new_tokens: int, num_layers: int) -> int:
    return int(_L().pkv_credit_pages(prompt_tokens, allowed_new_tokens, num_layers))


class Scheduler:
    """Admission and page allocation (C++ pkv_sched): continuous batching, or
    static batching (static=True: a new group only once the current one has
    finished)."""

    def __init__(self, num_pages: int, num_layers: int, max_blocks: int = 128, max_slots: int = 256,
                 static: bool = False):
        self._h = _L().pkv_sched_create(num_pages, num_layers, max_blocks, max_slots)
        if not self._h:
            raise PkvError(1, "pkv_sched_create")
        self.num_layers, self.max_blocks, self.max_slots = num_layers, max_blocks, max_slots
        if static:
            _check(_L().pkv_sched_set_mode(self._h, 1), "pkv_sched_set_mode")

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            _L().pkv_sched_destroy(h)
            self._h = None

    def submit(self, prompt_tokens: int, allowed_new_tokens: int):
        """Returns (status, request id); oversize requests give ERR_REQUEST_TOO_LARGE."""
        rid = ctypes.c_int(-1)
        st = _L().pkv_sched_submit(self._h, prompt_tokens, allowed_new_tokens, ctypes.byref(rid))
        if st not in (OK, ERR_REQUEST_TOO_LARGE):
            raise PkvError(st, "pkv_sched_submit")
        return st, rid.value

    def admit(self):
        buf = (ctypes.c_int * self.max_slots)()
        n = ctypes.c_int(0)
        _check(_L().pkv_sched_admit(self._h, buf, self.max_slots, ctypes.byref(n)), "pkv_sched_admit")
        return list(buf[:n.value])

    def grow(self, rid: int, new_len: int) -> int:
        st = _L().pkv_sched_grow(self._h, rid, new_len)
        if st not in (OK, ERR_POOL_EXHAUSTED):
            raise PkvError(st, "pkv_sched_grow")
        return st

    def finish(self, rid: int):
        _check(_L().pkv_sched_finish(self._h, rid), "pkv_sched_finish")

    def block_table(self, rid: int, layer: int):
        row = np.empty(self.max_blocks, np.int32)
        slot = ctypes.c_int(-1)
        _check(_L().pkv_sched_block_table(self._h, rid, layer, row.ctypes.data, ctypes.byref(slot)),
               "pkv_sched_block_table")
        return row, slot.value

    def stats(self):
        v = [ctypes.c_int(0) for _ in range(4)]
        _check(_L().pkv_sched_stats(self._h, *[ctypes.byref(x) for x in v]), "pkv_sched_stats")
        return dict(free=v[0].value, reserved=v[1].value, queued=v[2].value, running=v[3].value)

    def begin_step(self):
        """Grow every running request by one token (admission order); returns
        (ids, lengths after the step) as int32 arrays."""
        ids = np.empty(self.max_slots, np.int32)
        lens = np.empty(self.max_slots, np.int32)
        n = ctypes.c_int(0)
        st = _L().pkv_sched_begin_step(self._h, ids.ctypes.data, lens.ctypes.data, self.max_slots,
                                       ctypes.byref(n))
        _check(st, "pkv_sched_begin_step")
        return ids[:n.value].copy(), lens[:n.value].copy()

    def step_bytes(self, batch: int, max_len: int) -> int:
        return int(_L().pkv_sched_step_bytes(self._h, batch, max_len))

    def pack_step(self, ids, max_len: int, block) -> int:
        """Write the step block (lengths, then tables [L][B][P]) of requests
        `ids` into `block` (a contiguous uint8 host tensor or array); returns P."""
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        ptr = block.data_ptr() if isinstance(block, torch.Tensor) else block.ctypes.data
        nbytes = block.numel() if isinstance(block, torch.Tensor) else block.nbytes
        _check(_L().pkv_sched_pack_step(self._h, ids.ctypes.data, len(ids), int(max_len), ptr,
                                        nbytes), "pkv_sched_pack_step")
        return max(1, (int(max_len) + PAGE_TOKENS - 1) // PAGE_TOKENS)

    def events(self):
        n = _L().pkv_sched_event_count(self._h)
        out = []
        v = [ctypes.c_int(0) for _ in range(4)]
        for i in range(n):
            _check(_L().pkv_sched_event(self._h, i, *[ctypes.byref(x) for x in v]), "pkv_sched_event")
            out.append(tuple(x.value for x in v))
        return out


# --------------------------------------------------------------- decode step --

class DecodeStep:
    """One decode step over every layer, captured once into a CUDA graph.

    Per layer l (in order, as a model runs them), by default one fused call
        paged_gqa_decode_append(q[l], k[l], v[l], pool, block_tables[l],
                                seq_lens, out[l], cos, sin, q_out=q_rot[l])
    which appends token s of layer l at position seq_lens[s] - 1 and attends
    over seq_lens[s] tokens; the rotated queries are written only when the
    caller passes a q_rot buffer (the attention itself keeps them in
    registers: leaving the copy out saves about 0.2 us per layer at batch 32
    x 2048 on GB300).  With fused=False the same step runs as
        kv_append_rope(k[l], v[l], positions, block_tables[l], pool, cos, sin,
                       q_in=q[l], q_out=q_rot[l])
        paged_gqa_decode(q_rot[l], pool, block_tables[l], seq_lens, out[l], scale)
    (token s written at positions[s]).  The tensors are bound at construction: refresh
    their contents in place (new K/V/q, positions, lengths, tables) and call
    run().  Replaying the graph removes the per-call host cost, and the
    kernels' programmatic-dependent-launch edges overlap each launch with
    the previous kernel's tail.  With overlap_layers (the default) the decode
    kernel of layer l >= 1 also reads its tables and stages its first pages
    before layer l - 1's kernel has finished (early_kv), which requires the
    layers' block tables to name disjoint pages, as separate layers' caches
    do.  Layer 0 always waits for whatever ran before the step.

        pool          [num_pages, 2, 8, 16, 64] bf16
        block_tables  [L, S, max_blocks] int32
        seq_lens      [S] int32;  positions [S] int32
        k, v          [L, S, 8, 64] bf16;  q, out [L, S, 32, 64] bf16
    """

    def __init__(self, pool, block_tables, seq_lens, positions, k, v, q, out, rope_cos, rope_sin,
                 scale, max_seq_len=None, workspace=None, d_err=None, q_rot=None, compute=None,
                 use_graph=True, stream=None, fused=True, overlap_layers=True, schedule=None):
        self.L, self.S = block_tables.shape[0], block_tables.shape[1]
        self.t = dict(pool=pool, bt=block_tables, lens=seq_lens, pos=positions, k=k, v=v, q=q,
                      out=out, cos=rope_cos, sin=rope_sin)
        dev = pool.device
        self.workspace = alloc_workspace(self.S, dev) if workspace is None else workspace
        self.d_err = torch.zeros(1, dtype=torch.int32, device=dev) if d_err is None else d_err
        self.scale = float(scale)
        self.max_seq_len = max_seq_len
        self.compute = compute
        self.overlap = bool(overlap_layers)
        self.schedule = None if schedule is None else int(schedule)   # None: automatic
        # the fused kernel places each new token at seq_lens - 1 (positions unused)
        self.fused = fused and compute in (None, COMPUTE_TENSOR)
        # the rotated queries: kept by the fused step only in a buffer of the
        # caller's; the two-kernel step needs them (its decode reads them)
        self.q_rot = q_rot if (q_rot is not None or self.fused) else torch.empty_like(q)
        self._q_scratch = None  # the two-kernel timing graphs' rotated q on a fused step without q_rot
        self.launches_per_step = (1 if self.fused else 2) * self.L
        self._launch()                      # eager run: sets up kernels and descriptors
        torch.cuda.synchronize(dev)
        self.graph = None
        if use_graph:
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph, stream=stream):
                self._launch()

    def _launch(self, decode_only=False):
        t = self.t
        if self.fused and not decode_only:
            for l in range(self.L):
                paged_gqa_decode_append(t["q"][l], t["k"][l], t["v"][l], t["pool"], t["bt"][l],
                                        t["lens"], t["out"][l], t["cos"], t["sin"], self.scale,
                                        q_out=None if self.q_rot is None else self.q_rot[l],
                                        workspace=self.workspace,
                                        max_seq_len=self.max_seq_len, d_err=self.d_err,
                                        early_kv=int(self.overlap and l > 0),
                                        schedule=self.schedule)
            return
        q_rot = self._rotated()
        for l in range(self.L):
            if not decode_only:
                kv_append_rope(t["k"][l], t["v"][l], t["pos"], t["bt"][l], t["pool"], t["cos"],
                               t["sin"], q_in=t["q"][l], q_out=q_rot[l], d_err=self.d_err)
            # after kv_append_rope of the same layer the pages are not ready early
            paged_gqa_decode(q_rot[l], t["pool"], t["bt"][l], t["lens"], t["out"][l],
                             self.scale, workspace=self.workspace, max_seq_len=self.max_seq_len,
                             d_err=self.d_err, compute=self.compute,
                             early_kv=int(self.overlap and decode_only and l > 0),
                             schedule=self.schedule)

    def run(self):
        if self.graph is not None:
            self.graph.replay()
        else:
            self._launch()

    def _rotated(self):
        """The buffer the two-kernel form rotates q into: q_rot, else a
        scratch copy of q made on first use (outside any capture: the graph
        helpers below call this before capturing)."""
        if self.q_rot is not None:
            return self.q_rot
        if self._q_scratch is None:
            self._q_scratch = self.t["q"].clone()
        return self._q_scratch

    def append_only_graph(self):
        """A graph of just the L kv_append_rope calls of the step (tokens at
        `positions`, q rotated into the step's q_rot buffer, or a scratch one)."""
        t = self.t
        q_rot = self._rotated()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for l in range(self.L):
                kv_append_rope(t["k"][l], t["v"][l], t["pos"], t["bt"][l], t["pool"], t["cos"],
                               t["sin"], q_in=t["q"][l], q_out=q_rot[l], d_err=self.d_err)
        return g

    def decode_only_graph(self):
        """A graph of just the L decode calls (for timing the decode kernel)."""
        self._rotated()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self._launch(decode_only=True)
        return g

    def error(self) -> int:
        """Synchronise and return (and clear) the device error word."""
        return pkv_read_device_error(self.d_err)


class Int8DecodeStep:
    """One decode step over every layer on INT8 pages, captured into a CUDA graph.

    Per layer l:
        kv_append_rope_int8(k[l], v[l], positions, block_tables[l], kv_pool, cos, sin,
                            q_in=q[l], q_out=q_rot[l])
        paged_gqa_decode_int8(q_rot[l], kv_pool, block_tables[l], seq_lens, out[l], scale)
    (the fused form writes q_rot only when the caller passes one, as in DecodeStep)
    With fused=True each layer is one call
        paged_gqa_decode_append_int8(q[l], k[l], v[l], kv_pool, block_tables[l],
                                     seq_lens, out[l], cos, sin, q_out=q_rot[l])
    which places token s at seq_lens[s] - 1 (positions unused).  The default
    (fused=None) is the fused form, the faster one at every batch measured (on
    GB300 at 2048 tokens a sequence: 32 sequences 17.5 vs 23.1 us/layer, 256
    sequences 96.6 vs 108.4).  With
    overlap_layers (the default) layer l >= 1 reads its tables and stages its
    first pages before layer l - 1's kernel has finished, which requires the
    layers' block tables to name disjoint pages.  Tensors are bound at
    construction (refresh their contents in place and call run()), as for
    DecodeStep.

        kv_pool [num_pages, 8, 2176] uint8 (see new_int8_pool)
        block_tables [L, S, max_blocks] int32;  seq_lens, positions [S] int32
        k, v [L, S, 8, 64] bf16;  q, out [L, S, 32, 64] bf16
    """

    def __init__(self, kv_pool, block_tables, seq_lens, positions, k, v, q, out, rope_cos,
                 rope_sin, scale, max_seq_len=None, workspace=None, d_err=None, q_rot=None,
                 use_graph=True, stream=None, fused=None, overlap_layers=True):
        self.L, self.S = block_tables.shape[0], block_tables.shape[1]
        self.fused = True if fused is None else bool(fused)
        self.overlap = bool(overlap_layers)
        self.t = dict(pool=kv_pool, bt=block_tables, lens=seq_lens, pos=positions,
                      k=k, v=v, q=q, out=out, cos=rope_cos, sin=rope_sin)
        dev = kv_pool.device
        # the rotated queries, as for DecodeStep: kept by the fused step only
        # in a buffer of the caller's; the two-kernel step needs them
        self.q_rot = q_rot if (q_rot is not None or self.fused) else torch.empty_like(q)
        self._q_scratch = None  # the partial graphs' rotated q on a fused step without q_rot
        self.workspace = alloc_workspace(self.S, dev) if workspace is None else workspace
        self.d_err = torch.zeros(1, dtype=torch.int32, device=dev) if d_err is None else d_err
        self.scale = float(scale)
        self.max_seq_len = max_seq_len
        self.launches_per_step = (1 if self.fused else 2) * self.L
        self._launch()                      # eager run: sets up kernels and descriptors
        torch.cuda.synchronize(dev)
        self.graph = None
        if use_graph:
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph, stream=stream):
                self._launch()

    def _launch(self, append=True, decode=True):
        t = self.t
        if self.fused and append and decode:
            for l in range(self.L):
                paged_gqa_decode_append_int8(t["q"][l], t["k"][l], t["v"][l], t["pool"], t["bt"][l],
                                             t["lens"], t["out"][l], t["cos"], t["sin"], self.scale,
                                             q_out=None if self.q_rot is None else self.q_rot[l],
                                             workspace=self.workspace,
                                             max_seq_len=self.max_seq_len, d_err=self.d_err,
                                             early_kv=int(self.overlap and l > 0))
            return
        q_rot = self._rotated()
        for l in range(self.L):
            if append:
                kv_append_rope_int8(t["k"][l], t["v"][l], t["pos"], t["bt"][l], t["pool"],
                                    t["cos"], t["sin"], q_in=t["q"][l], q_out=q_rot[l],
                                    d_err=self.d_err)
            if decode:
                # a decode-only graph (timing) has no append between the layers:
                # layers >= 1 may stage their pages early, as in DecodeStep
                paged_gqa_decode_int8(q_rot[l], t["pool"], t["bt"][l], t["lens"], t["out"][l],
                                      self.scale, workspace=self.workspace,
                                      max_seq_len=self.max_seq_len, d_err=self.d_err,
                                      early_kv=int(self.overlap and not append and l > 0))

    def run(self):
        if self.graph is not None:
            self.graph.replay()
        else:
            self._launch()

    def _rotated(self):
        """As DecodeStep._rotated."""
        if self.q_rot is not None:
            return self.q_rot
        if self._q_scratch is None:
            self._q_scratch = self.t["q"].clone()
        return self._q_scratch

    def partial_graph(self, append: bool, decode: bool):
        """A graph of only the append calls or only the decode calls (for timing)."""
        self._rotated()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self._launch(append=append, decode=decode)
        return g

    def error(self) -> int:
        """Synchronise and return (and clear) the device error word."""
        return pkv_read_device_error(self.d_err)
