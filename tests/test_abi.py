"""The C-ABI library loads, exports every declared symbol, and validates arguments
on the host (no GPU needed: nothing here launches a kernel)."""
import ctypes
import glob
import os
import re

import numpy as np
import pytest

import oracle
import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def q():
    from prefill_dequant_gemv_gb300 import build as b
    b.build()
    import prefill_dequant_gemv_gb300 as q
    q.lib()
    return q


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(q\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(q):
    names = declared_functions()
    assert "qgemv" in names and "qg_pack_host" in names
    lib = ctypes.CDLL(q.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(q):
    assert q.qg_status_str(0) == "QG_OK"
    assert q.qg_status_str(6) == "QG_ERR_TIMEOUT"
    assert q.qg_status_str(99) == "QG_ERR_UNKNOWN"


@pytest.mark.parametrize("fmt,bpw", [(wl.MLX_AFFINE4_G64, 4.5), (wl.MXFP4, 4.25), (wl.NVFP4, 4.5), (wl.Q6K, 6.5625),
                                     (wl.Q5_0, 5.5), (wl.Q5_1, 6.0), (wl.Q5_K, 5.5)])
def test_packed_sizes_match_spec_and_bpw(q, fmt, bpw):
    for n, k in [(1024, 2048), (300, 768), (17408, 5120)]:
        assert q.qg_packed_sizes(fmt, n, k) == oracle.packed_sizes(fmt, n, k)
    c, s, a = q.qg_packed_sizes(fmt, 1024, 2048)
    assert (c + s + a) * 8 / (1024 * 2048) == bpw


def test_q6k_output_layer_is_1_04_gb(q):
    assert round(sum(q.qg_packed_sizes(wl.Q6K, 248320, 5120)) / 1e9, 2) == 1.04


@pytest.mark.parametrize("fmt", [wl.MLX_AFFINE4_G64, wl.MXFP4, wl.NVFP4, wl.Q6K, wl.Q5_0, wl.Q5_1, wl.Q5_K])
@pytest.mark.parametrize("shape", [(128, 256), (300, 768), (1, 256), (129, 512)])
def test_pack_round_trip_through_oracle_reader(q, fmt, shape):
    n, k = shape
    w = wl.weight(fmt, n, k, seed=n + k)
    c, s, a = q.qg_pack_host(fmt, n, k, w.codes, w.scales, w.aux)
    lc, ls, la = oracle.unpack(fmt, n, k, c, s, a if a.size else None)
    assert np.array_equal(lc, w.codes)
    assert np.array_equal(np.asarray(ls).view(np.uint8), np.asarray(w.scales).view(np.uint8))
    if w.aux is not None:
        assert np.array_equal(la.view(np.uint16), w.aux.view(np.uint16))
    # padding holds zero codes and zero scales
    fc, fs, fa = oracle.unpack(fmt, n, k, c, s, a if a.size else None, full=True)
    assert not fc[n:].any() and not fc[:, k:].any()


def test_pack_ragged_k_for_small_blocks(q):
    # NVFP4 K = 208 (13 blocks of 16), MXFP4, Q5_0 and Q5_1 K = 96 pad to whole 64-input groups
    for fmt, k in [(wl.NVFP4, 208), (wl.MXFP4, 96), (wl.Q5_0, 96), (wl.Q5_1, 160)]:
        w = wl.weight(fmt, 130, k, seed=3)
        c, s, a = q.qg_pack_host(fmt, 130, k, w.codes, w.scales, w.aux)
        lc, ls, la = oracle.unpack(fmt, 130, k, c, s)
        assert np.array_equal(lc, w.codes)
        assert np.array_equal(ls.view(np.uint8), np.asarray(w.scales).view(np.uint8))
        if w.aux is not None:
            assert np.array_equal(la.view(np.uint16), w.aux.view(np.uint16))


def test_pack_rejects_bad_input(q):
    w = wl.weight(wl.MLX_AFFINE4_G64, 128, 128, seed=1)
    bad = w.codes.copy()
    bad[3, 5] = 16
    with pytest.raises(q.QGError) as e:
        q.qg_pack_host(wl.MLX_AFFINE4_G64, 128, 128, bad, w.scales, w.aux)
    assert e.value.status == 1
    with pytest.raises(q.QGError):
        q.qg_packed_sizes(wl.NVFP4, 128, 100)  # K not a multiple of 16
    with pytest.raises(q.QGError):
        q.qg_packed_sizes(9, 128, 128)  # unknown format
    w5 = wl.weight(wl.Q5_K, 128, 256, seed=2)
    bad5 = w5.codes.copy()
    bad5[0, 0] = 32
    with pytest.raises(q.QGError):
        q.qg_pack_host(wl.Q5_K, 128, 256, bad5, w5.scales, w5.aux)  # 5-bit code above 31
    sm = w5.scales.copy()
    sm[1, 2, 1] = 64
    with pytest.raises(q.QGError):
        q.qg_pack_host(wl.Q5_K, 128, 256, w5.codes, sm, w5.aux)  # 6-bit minimum above 63
    with pytest.raises(q.QGError):
        q.qg_packed_sizes(wl.Q5_K, 128, 128)  # K not a multiple of 256


def _desc(q, **kw):
    d = dict(fmt=wl.NVFP4, reserved=0, n=256, k=256, codes=0x1000, scales=0x2000, aux=None, tensor_scale=1.0,
             reserved2=0.0)
    d.update(kw)
    return q.qg_weight(**d)


@pytest.mark.parametrize("kw,status", [
    (dict(fmt=7), 1), (dict(k=100), 1), (dict(codes=None), 1), (dict(reserved=1), 1),
    (dict(fmt=wl.MXFP4, tensor_scale=0.5), 1), (dict(fmt=wl.Q6K, k=512, aux=None), 1),
    (dict(codes=0x1008), 3),
])
def test_qgemv_host_validation(q, kw, status):
    w = _desc(q, **kw)
    st = q.lib().qgemv(ctypes.byref(w), 0x3000, 1, 256, None, 0, 0x4000, 256, 0x5000, 1 << 20, None)
    assert st == status


def test_qgemv_rejects_bad_rows_and_strides(q):
    w = _desc(q)
    L = q.lib()
    assert L.qgemv(ctypes.byref(w), 0x3000, 0, 256, None, 0, 0x4000, 256, 0x5000, 1 << 20, None) == 2
    assert L.qgemv(ctypes.byref(w), 0x3000, 5, 256, None, 0, 0x4000, 256, 0x5000, 1 << 20, None) == 2
    assert L.qgemv(ctypes.byref(w), 0x3000, 1, 260, None, 0, 0x4000, 256, 0x5000, 1 << 20, None) == 3
    assert L.qgemv(ctypes.byref(w), 0x3008, 1, 256, None, 0, 0x4000, 256, 0x5000, 1 << 20, None) == 3
    assert L.qgemv(ctypes.byref(w), None, 1, 256, None, 0, 0x4000, 256, 0x5000, 1 << 20, None) == 1
    assert L.qgemv(ctypes.byref(w), 0x3000, 1, 128, None, 0, 0x4000, 256, 0x5000, 1 << 20, None) == 1


def _moe_desc(q, **kw):
    d = dict(fmt=wl.MXFP4, n_experts=8, hidden=256, ffn=128, gu_codes=0x10000, gu_scales=0x20000, gu_aux=None,
             dn_codes=0x30000, dn_scales=0x40000, dn_aux=None, tensor_scale=1.0, has_shared=0)
    d.update(kw)
    return q.qg_moe_layer(**d)


def test_qgemm_grouped_host_validation(q):
    """Argument errors of the staged MoE call come back before any device work."""
    L = q.lib()
    m = _moe_desc(q)
    args = dict(stage=q.QG_MOE_GATE_UP_SWIGLU, inp=0x3000, t=4, ldi=256, topk=2, w=0x6000, gate=None, rws=0x7000,
                out=0x8000, ldo=128, ws=0x9000, wsb=1 << 24)

    def call(layer=m, **kw):
        a = dict(args)
        a.update(kw)
        return L.qgemm_grouped(ctypes.byref(layer), a["stage"], a["inp"], a["t"], a["ldi"], a["topk"], a["w"],
                               a["gate"], a["rws"], a["out"], a["ldo"], a["ws"], a["wsb"], None)

    assert call(stage=3) == 1                                   # unknown stage
    assert call(stage=0) == 1
    assert call(inp=None) == 1
    assert call(stage=q.QG_MOE_DOWN_COMBINE, w=None, ldi=128, ldo=256) == 1  # the combine needs topk_w
    assert call(ldi=128) == 1                                   # gate/up input narrower than H
    assert call(stage=q.QG_MOE_DOWN_COMBINE, ldi=64, ldo=256) == 1  # down input narrower than F
    assert call(inp=0x3008) == 3                                # misaligned
    assert call(ldo=132) == 3                                   # leading dimension not a multiple of 8
    assert call(topk=9) == 1                                    # more than the experts
    assert call(layer=_moe_desc(q, n_experts=32), topk=17) == 2  # above the router's limit
    assert call(t=0) == 1
    assert call(gate=0xA000) == 1                               # gate logits without a shared expert
    assert call(layer=_moe_desc(q, fmt=wl.Q5_0)) == 2           # the 5-bit formats run on the dense paths only
    # the prefill chain (more than 4 tokens) pairs gate and up rows in one 128-row tile
    assert call(layer=_moe_desc(q, ffn=96), t=8, ldo=96) == 2
    assert call(layer=_moe_desc(q, ffn=96), t=8, stage=q.QG_MOE_DOWN_COMBINE, ldi=96, ldo=256) == 2
    sh = _moe_desc(q, has_shared=1,
                   shared_gate_up=q.qg_weight(fmt=wl.MXFP4, n=256, k=256, codes=0x50000, scales=0x51000,
                                              tensor_scale=1.0),
                   shared_down=q.qg_weight(fmt=wl.MXFP4, n=256, k=128, codes=0x52000, scales=0x53000,
                                           tensor_scale=1.0))
    assert call(layer=sh, gate=0xA002) == 3                     # misaligned gate logits
    assert L.qgemm_grouped_workspace_size(ctypes.byref(m), 4, 2, 3) == 0


def test_qmoe_forward_host_validation(q):
    """Argument errors of the router + FFN call come back before any device work."""
    L = q.lib()
    m = _moe_desc(q)
    args = dict(x=0x3000, t=4, ldx=256, lg=0x4000, topk=2, gate=None, ids=0x5000, w=0x6000, rws=0x7000,
                rwsb=1 << 20, out=0x8000, ldo=256, ws=0x9000, wsb=1 << 26)

    def call(layer=m, **kw):
        a = dict(args)
        a.update(kw)
        return L.qmoe_forward(ctypes.byref(layer), a["x"], a["t"], a["ldx"], a["lg"], a["topk"], a["gate"], a["ids"],
                              a["w"], a["rws"], a["rwsb"], a["out"], a["ldo"], a["ws"], a["wsb"], None)

    assert call(lg=None) == 1                      # logits required
    assert call(ids=None) == 1
    assert call(t=0) == 1
    assert call(topk=9) == 1                       # more than the experts
    assert call(gate=0xA000) == 1                  # gate logits without a shared expert
    assert call(lg=0x4004) == 3                    # misaligned logits
    assert call(ldo=128) == 1                      # output narrower than H
    assert call(rwsb=16) == 4                      # router workspace too small
    assert call(layer=_moe_desc(q, fmt=wl.Q6K)) == 1  # Q6_K layer without aux
    assert call(layer=_moe_desc(q, fmt=wl.Q5_K)) == 2  # the 5-bit formats run on the dense paths only


def test_quant_act_nvfp4_host_validation(q):
    """Argument errors of the activation quantiser come back before anything is launched."""
    L = q.lib()
    args = dict(x=0x3000, m=4, k=256, ldx=256, a=1.0, c=0x4000, ldc=128, s=0x5000, lds=16, xe=0x6000, lde=256)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return L.qg_quant_act_nvfp4(a["x"], a["m"], a["k"], a["ldx"], a["a"], a["c"], a["ldc"], a["s"], a["lds"],
                                    a["xe"], a["lde"], None)
    assert call(x=None) == 1 and call(m=0) == 1 and call(k=250) == 1 and call(k=0) == 1
    assert call(a=0.0) == 1 and call(a=-1.0) == 1 and call(a=float("inf")) == 1 and call(a=float("nan")) == 1
    assert call(ldx=128) == 1 and call(ldc=64) == 1 and call(lds=8) == 1 and call(lde=128) == 1
    assert call(x=0x3008) == 3 and call(ldx=260) == 3 and call(c=0x4008) == 3 and call(ldc=132) == 3
    assert call(xe=0x6008) == 3 and call(lde=260) == 3
    assert call(m=1 << 27) == 2  # 2^31 blocks of 16: beyond the kernel's 32-bit block index


def test_qgemm_w4a4_host_validation(q):
    """The W4A4 GEMM makes every check qgemm makes (plus its own) before launching."""
    L = q.lib()
    w = _desc(q, tensor_scale=0.5)

    def call(wd=w, x=0x3000, m=8, ldx=256, a=1.0, y=0x4000, ldy=256, ws=0x5000, wsb=1 << 20):
        return L.qgemm_w4a4(ctypes.byref(wd), x, m, ldx, a, None, 0, y, ldy, ws, wsb, None)
    assert call(wd=_desc(q, fmt=wl.MXFP4)) == 2 and call(m=0) == 2
    assert call(x=None) == 1 and call(a=0.0) == 1 and call(a=float("nan")) == 1
    assert call(wd=_desc(q, tensor_scale=1e30), a=1e30) == 1  # the product overflows fp32
    assert call(ldx=128) == 1 and call(ldy=128) == 1
    assert call(x=0x3008) == 3 and call(y=0x4008) == 3 and call(ldx=260) == 3
    # 8 rows (the FP4 GEMM): status header, then codes 8 x 128 bytes from offset 256, then
    # E4M3 scales 8 x 16 bytes from the next 256-byte boundary (1280)
    assert q.qgemm_w4a4_workspace_size(wl.NVFP4, 256, 256, 8) == 1280 + 8 * 16
    assert call(wsb=1000) == 4
    assert q.qgemm_w4a4_workspace_size(wl.NVFP4, 256, 1000, 8) == 0  # K not a multiple of 16
    assert q.qgemm_w4a4_workspace_size(wl.MXFP4, 256, 256, 8) == 0
    assert q.qgemm_w4a4_workspace_size(wl.NVFP4, 256, 256, 0) == 0
