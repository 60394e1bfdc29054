"""Oracle-backed stand-ins for the library's kernel calls, for CPU tests of
the host logic that drives them (serving.ContinuousBatcher).

Each stand-in takes the binding's arguments (CPU tensors), checks the
contract the host side must keep (dtypes, shapes, contiguity, int32 indices,
max_seq_len an upper bound of the lengths) and computes through the FP64
oracle, writing pools and outputs in place as the kernels do.  Test
infrastructure only: nothing outside tests/ imports it.
"""
import numpy as np
import torch

import workloads as W
from oracle import int8_kv as OI, paged_kv as OP

ERR_DEVICE_INDEX = 6


def _bits(t):
    return W.bf16_bits(t)


def _bf16(b, like):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).view(like.shape)


def _flag(err, d_err):
    if err and d_err is not None and int(d_err[0]) == 0:
        d_err[0] = ERR_DEVICE_INDEX


def _check_tables(block_tables, seq_lens=None, max_seq_len=None):
    assert block_tables.dtype == torch.int32 and block_tables.dim() == 2
    assert block_tables.is_contiguous()
    if seq_lens is not None:
        assert seq_lens.dtype == torch.int32 and seq_lens.is_contiguous()
        if max_seq_len is not None and seq_lens.numel():
            assert int(seq_lens.max()) <= max_seq_len, "max_seq_len below a length"


def _rows(t, width):
    assert t.dtype == torch.bfloat16 and t.is_contiguous()
    return _bits(t).reshape(-1, width, W.HEAD_DIM)


def kv_append_rope(k, v, positions, block_tables, kv_pool, rope_cos, rope_sin, token_seq=None,
                   q_in=None, q_out=None, d_err=None, max_blocks=None, stream=None):
    _check_tables(block_tables)
    assert positions.dtype == torch.int32 and kv_pool.dtype == torch.bfloat16
    bt = block_tables.numpy()[:, :max_blocks] if max_blocks else block_tables.numpy()
    pool, qr, err = OP.append_rope(_bits(kv_pool), _rows(k, 8), _rows(v, 8), positions.numpy(),
                                   None if token_seq is None else token_seq.numpy(), bt,
                                   rope_cos.numpy(), rope_sin.numpy(),
                                   None if q_in is None else _rows(q_in, 32))
    kv_pool.copy_(_bf16(pool, kv_pool))
    if q_in is not None:
        q_out.copy_(_bf16(qr, q_out))
    _flag(err, d_err)


def kv_append_rope_int8(k, v, positions, block_tables, kv_pool, rope_cos, rope_sin,
                        token_seq=None, q_in=None, q_out=None, d_err=None, max_blocks=None,
                        stream=None):
    _check_tables(block_tables)
    assert positions.dtype == torch.int32 and kv_pool.dtype == torch.uint8
    bt = block_tables.numpy()[:, :max_blocks] if max_blocks else block_tables.numpy()
    codes, scales = OI.unpack_pages(kv_pool.numpy())
    codes, scales, qr, err = OI.append_rope_int8(
        codes, scales, _rows(k, 8), _rows(v, 8), positions.numpy(),
        None if token_seq is None else token_seq.numpy(), bt, rope_cos.numpy(), rope_sin.numpy(),
        None if q_in is None else _rows(q_in, 32))
    kv_pool.copy_(torch.from_numpy(OI.pack_pages(codes, scales)))
    if q_in is not None:
        q_out.copy_(_bf16(qr, q_out))
    _flag(err, d_err)


def kv_append_rope_layers(k, v, positions, block_tables, kv_pool, rope_cos, rope_sin,
                          token_seq=None, stage=None, d_err=None, max_blocks=None, stream=None):
    assert len(k) == len(v) and len(k) > 0
    assert block_tables.dtype == torch.int32 and block_tables.dim() == 3
    assert block_tables.stride(2) == 1 and block_tables.shape[0] >= len(k)
    assert all(t.device == k[0].device for t in list(k) + list(v))
    append = kv_append_rope_int8 if kv_pool.dtype == torch.uint8 else kv_append_rope
    for l in range(len(k)):
        append(k[l], v[l], positions, block_tables[l].contiguous(), kv_pool, rope_cos, rope_sin,
               token_seq=token_seq, d_err=d_err, max_blocks=max_blocks)


def _write_out(out, o):
    out.copy_(torch.from_numpy(o).to(torch.bfloat16).view(out.shape))


def paged_gqa_decode(q, kv_pool, block_tables, seq_lens, out, scale, workspace=None,
                     max_seq_len=None, d_err=None, max_blocks=None, **kw):
    _check_tables(block_tables, seq_lens, max_seq_len)
    q_b = _rows(q, 32)
    o, err = OP.decode(q_b, _bits(kv_pool), block_tables.numpy()[:q_b.shape[0]],
                       seq_lens.numpy(), scale)
    _write_out(out, o)
    _flag(err, d_err)


def paged_gqa_decode_int8(q, kv_pool, block_tables, seq_lens, out, scale, workspace=None,
                          max_seq_len=None, d_err=None, max_blocks=None, **kw):
    _check_tables(block_tables, seq_lens, max_seq_len)
    q_b = _rows(q, 32)
    codes, scales = OI.unpack_pages(kv_pool.numpy())
    o, err = OI.decode_int8(q_b, codes, scales, block_tables.numpy()[:q_b.shape[0]],
                            seq_lens.numpy(), scale)
    _write_out(out, o)
    _flag(err, d_err)


def paged_gqa_decode_append(q, k_new, v_new, kv_pool, block_tables, seq_lens, out, rope_cos,
                            rope_sin, scale, q_out=None, workspace=None, max_seq_len=None,
                            d_err=None, **kw):
    _check_tables(block_tables, seq_lens, max_seq_len)
    q_b = _rows(q, 32)
    pool, qr, o, err = OP.decode_step(_bits(kv_pool), q_b, _rows(k_new, 8), _rows(v_new, 8),
                                      block_tables.numpy()[:q_b.shape[0]], seq_lens.numpy(),
                                      rope_cos.numpy(), rope_sin.numpy(), scale)
    kv_pool.copy_(_bf16(pool, kv_pool))
    if q_out is not None:
        q_out.copy_(_bf16(qr, q_out))
    _write_out(out, o)
    _flag(err, d_err)


def paged_gqa_decode_append_int8(q, k_new, v_new, kv_pool, block_tables, seq_lens, out, rope_cos,
                                 rope_sin, scale, q_out=None, workspace=None, max_seq_len=None,
                                 d_err=None, **kw):
    _check_tables(block_tables, seq_lens, max_seq_len)
    q_b = _rows(q, 32)
    codes, scales = OI.unpack_pages(kv_pool.numpy())
    codes, scales, qr, o, err = OI.decode_step_int8(
        codes, scales, q_b, _rows(k_new, 8), _rows(v_new, 8),
        block_tables.numpy()[:q_b.shape[0]], seq_lens.numpy(), rope_cos.numpy(),
        rope_sin.numpy(), scale)
    kv_pool.copy_(torch.from_numpy(OI.pack_pages(codes, scales)))
    if q_out is not None:
        q_out.copy_(_bf16(qr, q_out))
    _write_out(out, o)
    _flag(err, d_err)


def paged_gqa_decode_append_layers(q, k_new, v_new, kv_pool, block_tables, seq_lens, out,
                                   rope_cos, rope_sin, scale, workspace, max_seq_len=None,
                                   d_err=None, stream=None, q_out=None, early_kv=1,
                                   host_stage=None, dev_stage=None, check=True):
    assert q.dim() == 4 and block_tables.dim() == 3 and block_tables.shape[0] == q.shape[0]
    assert (host_stage is None) == (dev_stage is None) and early_kv in (0, 1)
    if host_stage is not None:       # the step block's copy comes first
        assert host_stage.dtype == torch.uint8 and dev_stage.numel() >= host_stage.numel()
        dev_stage[:host_stage.numel()].copy_(host_stage)
    step = paged_gqa_decode_append_int8 if kv_pool.dtype == torch.uint8 else paged_gqa_decode_append
    for l in range(q.shape[0]):
        step(q[l], k_new[l], v_new[l], kv_pool, block_tables[l], seq_lens, out[l], rope_cos,
             rope_sin, scale, q_out=None if q_out is None else q_out[l], workspace=workspace,
             max_seq_len=max_seq_len, d_err=d_err)


def alloc_workspace(num_seqs, device):
    return torch.zeros(16, dtype=torch.uint8)


def pkv_read_device_error(d_err, clear=True, stream=None):
    code = int(d_err[0])
    if clear:
        d_err[0] = 0
    return code


NAMES = ("kv_append_rope", "kv_append_rope_int8", "kv_append_rope_layers",
         "paged_gqa_decode", "paged_gqa_decode_int8",
         "paged_gqa_decode_append", "paged_gqa_decode_append_int8",
         "paged_gqa_decode_append_layers", "alloc_workspace",
         "pkv_read_device_error")


def patch_serving(monkeypatch):
    """Point serving's kernel calls (the ones it imports) at the stand-ins above."""
    import paged_kv_gqa_append_gb300.serving as S
    g = globals()
    patched = [n for n in NAMES if hasattr(S, n)]
    for n in patched:
        monkeypatch.setattr(S, n, g[n])
    assert "paged_gqa_decode_append_layers" in patched and "paged_gqa_decode" in patched
