"""Binding-level checks that need no GPU: the C calls the Python binding
makes, recorded by a stand-in for the loaded library.

paged_gqa_decode_append_layers makes one call of the C function of the same
name; the per-layer pointers that function derives (base + l x the layer's
bytes, tables base + l x bt_layer_stride) must be exactly the arguments that
L calls of the per-layer binding pass, so that the per-layer path's GPU
parity carries over (the GPU tests also compare the two bit for bit).
"""
import ctypes
import types

import pytest
import torch

import paged_kv_gqa_append_gb300 as pkv

BF16, I32 = torch.bfloat16, torch.int32


class Recorder:
    """Stands in for libpkv.so: records each call's entry point and arguments
    (pointers as integers, option structs as field tuples) and returns OK."""

    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def call(*args):
            self.calls.append((name, tuple(self._norm(a) for a in args)))
            return pkv.OK
        return call

    @staticmethod
    def _norm(a):
        if isinstance(a, ctypes.c_void_p):
            return a.value
        if type(a).__name__ == "CArgObject":
            obj = a._obj
            return tuple(getattr(obj, f) for f, _ in obj._fields_)
        return a

    def take(self):
        out, self.calls = self.calls, []
        return out


def tensors(int8, L=3, S=5, S_rows=7, row_stride=128):
    pool = (pkv.new_int8_pool(11, "cpu") if int8
            else torch.zeros((11, 2, 8, 16, 64), dtype=BF16))
    return dict(
        q=torch.zeros((L, S, 32, 64), dtype=BF16), k=torch.zeros((L, S, 8, 64), dtype=BF16),
        v=torch.zeros((L, S, 8, 64), dtype=BF16), out=torch.zeros((L, S, 32, 64), dtype=BF16),
        bt=torch.zeros((L, S_rows, row_stride), dtype=I32), lens=torch.zeros(S, dtype=I32),
        cos=torch.zeros((64, 32)), sin=torch.zeros((64, 32)),
        ws=torch.zeros(4096, dtype=torch.uint8), err=torch.zeros(1, dtype=I32), pool=pool)


@pytest.fixture
def rec(monkeypatch):
    r = Recorder()
    monkeypatch.setattr(pkv, "_L", lambda: r)
    return r


STREAM = types.SimpleNamespace(cuda_stream=0x1234)


@pytest.mark.parametrize("int8", [False, True])
@pytest.mark.parametrize("max_seq_len", [None, 77])
def test_layers_call_derives_the_per_layer_calls(rec, int8, max_seq_len):
    t = tensors(int8)
    L, S = t["q"].shape[:2]
    per_layer = pkv.paged_gqa_decode_append_int8 if int8 else pkv.paged_gqa_decode_append
    for l in range(L):
        per_layer(t["q"][l], t["k"][l], t["v"][l], t["pool"], t["bt"][l], t["lens"], t["out"][l],
                  t["cos"], t["sin"], 0.125, workspace=t["ws"], max_seq_len=max_seq_len,
                  d_err=t["err"], stream=STREAM)
    want = rec.take()
    pkv.paged_gqa_decode_append_layers(t["q"], t["k"], t["v"], t["pool"], t["bt"], t["lens"],
                                       t["out"], t["cos"], t["sin"], 0.125, t["ws"],
                                       max_seq_len=max_seq_len, d_err=t["err"], stream=STREAM)
    got = rec.take()
    assert len(got) == 1 and got[0][0] == "paged_gqa_decode_append_layers"
    (q, k, v, q_out, out, nl, ns, cos, sin, max_pos, pool, npages, i8, bt, bt_ls, bt_rs, mb, lens,
     msl, scale, ws, wsb, err, stream, early, hst, dst, sb) = got[0][1]
    assert (nl, ns, i8, early, hst, dst, sb, q_out) == (L, S, int(int8), 1, None, None, 0, None)
    qb, kb = S * 32 * 64 * 2, S * 8 * 64 * 2
    name = "paged_gqa_decode_append_int8" if int8 else "paged_gqa_decode_append"
    for l, (fn, a) in enumerate(want):
        assert fn == name
        # per-layer arguments: q, k, v, cos, sin, max_pos, pool, pages, bt, stride, max_blocks,
        # lens, S, max_seq_len, q_out, out, scale, ws, ws bytes, d_err, stream, opts
        assert a[0] == q + l * qb and a[1] == k + l * kb and a[2] == v + l * kb
        assert a[3:8] == (cos, sin, max_pos, pool, npages)
        assert a[8] == bt + 4 * l * bt_ls and (a[9], a[10]) == (bt_rs, mb)
        assert (a[11], a[12], a[13], a[14]) == (lens, S, msl, None)
        assert a[15] == out + l * qb
        assert a[16:21] == (scale, ws, wsb, err, stream)
        # default options, automatic schedule (the native call sets early_kv on
        # layers >= 1 itself)
        assert a[21] == (pkv.COMPUTE_TENSOR, 0, 0, 0, 0, 0, pkv.SCHEDULE_AUTO, 0, 0, 0)


@pytest.mark.parametrize("bad", ["out_shape", "kv_layers", "tables_layers", "tables_rows",
                                 "lens", "not_4d", "strided"])
def test_layers_call_rejects_bad_shapes_before_any_call(rec, bad):
    t = tensors(False)
    if bad == "out_shape":
        t["out"] = t["out"][:, :4].contiguous()
    elif bad == "kv_layers":
        t["k"] = t["k"][:2].contiguous()
    elif bad == "tables_layers":
        t["bt"] = t["bt"][:2].contiguous()
    elif bad == "tables_rows":
        t["bt"] = t["bt"][:, :4].contiguous()
    elif bad == "lens":
        t["lens"] = t["lens"][:4].contiguous()
    elif bad == "not_4d":
        t["q"] = t["q"].reshape(15, 32, 64)
    elif bad == "strided":
        t["q"] = torch.zeros((5, 3, 32, 64), dtype=BF16).transpose(0, 1)
    with pytest.raises((ValueError, TypeError)):
        pkv.paged_gqa_decode_append_layers(t["q"], t["k"], t["v"], t["pool"], t["bt"], t["lens"],
                                           t["out"], t["cos"], t["sin"], 0.125, t["ws"],
                                           d_err=t["err"], stream=STREAM)
    assert rec.calls == []


def prompt_tensors(int8, L=3, P=20):
    t = tensors(int8, L=L)
    t["pk"] = [torch.full((P, 8, 64), float(l), dtype=BF16) for l in range(L)]
    t["pv"] = [torch.full((P, 8, 64), -float(l), dtype=BF16) for l in range(L)]
    t["pos"] = torch.arange(P, dtype=I32)
    t["row0"] = torch.zeros(P, dtype=I32)
    t["stage"] = torch.zeros(2 * P * 1024, dtype=torch.uint8)
    return t


@pytest.mark.parametrize("int8", [False, True])
def test_prompt_layers_call_marshals_the_row_view(rec, int8):
    # host rows (the pool here is on the CPU too, so the rows count as host
    # memory): one native call with the per-layer pointer arrays, the layer
    # stride of the full table, the one-row view's row and its row stride
    L, P, slot = 3, 20, 4
    t = prompt_tensors(int8, L=L, P=P)
    view = t["bt"][:, slot:slot + 1]
    pkv.kv_append_rope_layers(t["pk"], t["pv"], t["pos"], view, t["pool"], t["cos"], t["sin"],
                              token_seq=t["row0"], stage=t["stage"], d_err=t["err"], stream=STREAM)
    (name, a), = rec.take()
    assert name == "kv_append_rope_layers"
    ks, vs = [x for x in a[0]], [x for x in a[1]]
    assert ks == [x.data_ptr() for x in t["pk"]] and vs == [x.data_ptr() for x in t["pv"]]
    assert a[2:9] == (L, 1, t["stage"].data_ptr(), t["stage"].numel(), t["pos"].data_ptr(),
                      t["row0"].data_ptr(), P)
    assert a[9] == view.data_ptr() == t["bt"].data_ptr() + 4 * slot * 128
    assert a[10:14] == (7 * 128, 1, 128, 128)        # layer stride, rows, row stride, max_blocks
    assert a[14:17] == (t["pool"].data_ptr(), 11, int(int8))


@pytest.mark.parametrize("bad", ["layers", "rows", "tables_2d", "tables_strided", "tables_layers",
                                 "no_stage", "short_stage"])
def test_prompt_layers_call_rejects_bad_arguments(rec, bad):
    t = prompt_tensors(False)
    bt, stage = t["bt"], t["stage"]
    if bad == "layers":
        t["pv"] = t["pv"][:2]
    elif bad == "rows":
        t["pk"][1] = t["pk"][1][:10].contiguous()
    elif bad == "tables_2d":
        bt = bt[0]
    elif bad == "tables_strided":
        bt = bt.transpose(1, 2)
    elif bad == "tables_layers":
        bt = bt[:2]
    elif bad == "no_stage":
        stage = None
    elif bad == "short_stage":
        stage = stage[:1000]
    with pytest.raises((ValueError, TypeError)):
        pkv.kv_append_rope_layers(t["pk"], t["pv"], t["pos"], bt, t["pool"], t["cos"], t["sin"],
                                  token_seq=t["row0"], stage=stage, d_err=t["err"], stream=STREAM)
    assert rec.calls == []
