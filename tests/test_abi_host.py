"""Host-side tests of the C ABI (no GPU needed): the library builds and loads, exports every
entry point of include/lora_mlp.h, its NF4 table equals the oracle's bit for bit, and argument
errors are reported before anything reaches the device."""
import ctypes

import numpy as np
import pytest

from bwd_lora_mlp_gb300 import build as B
from bwd_lora_mlp_gb300 import lib as L
from oracle import nf4 as onf4


@pytest.fixture(scope="module")
def so():
    B.build()
    return L.load()


def test_exports_every_header_symbol(so):
    names = L.header_symbols()
    assert len(names) == 32
    for n in names:
        assert hasattr(so, n), n
    assert set(names) == set(L._SIGS)


def test_build_is_keyed_on_source_content(so, tmp_path):
    """The built library is reused only while the digest stored beside it matches the sources and
    flags; any other digest (other sources, other flags, or none at all) means a rebuild."""
    assert B.up_to_date()
    with open(B.DIGEST) as f:
        assert f.read().strip() == B.source_digest()
    assert B.source_digest(["-DLM_SOMETHING_ELSE"]) != B.source_digest()
    assert not B.up_to_date(["-DLM_SOMETHING_ELSE"])


def test_codebook_matches_oracle_bitwise(so):
    cb = np.array(L.lm_nf4_codebook(), dtype=np.float32)
    assert np.array_equal(cb.view(np.uint32), onf4.codebook().view(np.uint32))


def _size(fn, *args):
    out = ctypes.c_size_t(0)
    st = L.call_status(fn, *args, ctypes.byref(out))
    return st, out.value


def test_size_queries():
    st, s1 = _size("lora_mlp_workspace_size", 512, 256, 704, 8)
    assert st == L.LM_OK and s1 > 2 * 512 * 704 * 2
    st, s2 = _size("lora_mlp_workspace_size", 1024, 256, 704, 8)
    assert st == L.LM_OK and s2 > s1
    assert _size("lora_mlp_workspace_size", 512, 250, 704, 8)[0] == L.LM_ERR_SHAPE
    assert _size("lora_mlp_workspace_size", 512, 256, 704, 12)[0] == L.LM_ERR_SHAPE
    assert _size("lora_mlp_workspace_size", 512, 256, 704, 72)[0] == L.LM_ERR_SHAPE
    assert _size("lora_mlp_workspace_size", -1, 256, 704, 8)[0] == L.LM_ERR_SHAPE
    assert L.call_status("lora_mlp_saved_size", 512, 8, None) == L.LM_ERR_NULL
    for fn, args in (("lora_mlp_saved_size", (0, 16)), ("lora_qkv_saved_size", (100, 16)),
                     ("lora_o_saved_size", (100, 64)), ("lora_qkv_workspace_size", (100, 256, 256, 64, 64, 16)),
                     ("lora_o_workspace_size", (100, 256, 128, 16))):
        st, v = _size(fn, *args)
        assert st == L.LM_OK and v > 0, fn


# ---------------------------------------------------------------------------- fake device pointers
# Validation runs on the host before any CUDA call, so distinct aligned integers stand in for
# device buffers; none is ever dereferenced.

class Fake:
    def __init__(self):
        self.next = 1 << 32

    def __call__(self, nbytes):
        p = self.next
        self.next += (int(nbytes) + 4095) // 4096 * 4096 + 4096
        return p


def _lora(fake, din, dout, r, s=2.0):
    w = L.lm_weight()
    w.kind, w.rows, w.cols = L.LM_WEIGHT_BF16, dout, din
    w.w = fake(din * dout * 2)
    x = L.lm_lora()
    x.W, x.A, x.B, x.r, x.s = w, fake(r * din * 2), fake(dout * r * 2), r, s
    return x


def _mlp_args(T=512, d=256, n=704, r=8, **over):
    f = Fake()
    a = dict(T=T, d=d, n=n, act=L.LM_ACT_SWIGLU, X=f(T * d * 2), gate=_lora(f, d, n, r), up=_lora(f, d, n, r),
             down=_lora(f, n, d, r), y=f(T * d * 2), e=f(T * n * 2), u=f(T * n * 2), h=f(T * n * 2))
    a["saved_bytes"] = _size("lora_mlp_saved_size", T, r)[1]
    a["saved"] = f(a["saved_bytes"])
    a["ws_bytes"] = _size("lora_mlp_workspace_size", T, d, n, r)[1]
    a["ws"] = f(a["ws_bytes"])
    a.update(over)
    return a


def _fwd(a):
    return L.call_status("lora_mlp_fwd", a["T"], a["d"], a["n"], a["act"], a["X"], ctypes.byref(a["gate"]),
                         ctypes.byref(a["up"]), ctypes.byref(a["down"]), a["y"], a["e"], a["u"], a["h"],
                         a["saved"], a["saved_bytes"], a["ws"], a["ws_bytes"], None)


def test_mlp_fwd_argument_errors(so):
    assert _fwd(_mlp_args(X=None)) == L.LM_ERR_NULL
    a = _mlp_args()
    assert _fwd(dict(a, X=a["X"] + 2)) == L.LM_ERR_ALIGN
    assert _fwd(dict(a, X=a["X"] + 16)) == L.LM_ERR_ALIGN  # 32-byte rule
    assert _fwd(dict(a, y=a["X"])) == L.LM_ERR_ALIAS                       # in-place not offered
    assert _fwd(dict(a, h=a["e"] + 64)) == L.LM_ERR_ALIAS                  # two outputs overlap
    assert _fwd(dict(a, ws_bytes=a["ws_bytes"] - 1)) == L.LM_ERR_WORKSPACE
    assert _fwd(dict(a, saved_bytes=16)) == L.LM_ERR_WORKSPACE
    assert _fwd(dict(a, act=7)) == L.LM_ERR_DTYPE
    assert _fwd(dict(a, d=250)) == L.LM_ERR_SHAPE
    b = _mlp_args()
    b["up"].r = 16
    assert _fwd(b) == L.LM_ERR_SHAPE                                       # ranks differ
    c = _mlp_args()
    c["down"].W.rows = 128
    assert _fwd(c) == L.LM_ERR_SHAPE                                       # W shape mismatch
    k = _mlp_args()
    k["gate"].W.kind = 5
    assert _fwd(k) == L.LM_ERR_DTYPE
    z = _mlp_args()
    z["gate"].s = float("nan")
    assert _fwd(z) == L.LM_ERR_SHAPE
    assert "gate.s" in L.last_error()
    t = _mlp_args()
    t["up"].ab_dtype = 7                                                   # neither bf16 nor fp32 A/B
    assert _fwd(t) == L.LM_ERR_DTYPE
    assert "up.ab_dtype" in L.last_error()


def test_empty_token_count_is_a_no_op(so):
    a = _mlp_args(T=0)
    assert _fwd(a) == L.LM_OK


def test_without_device_reports_cuda_error(so):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    st = _fwd(_mlp_args())
    assert st in (L.LM_ERR_CUDA, L.LM_ERR_UNSUPPORTED)
    assert L.last_error()


def test_nf4_argument_errors(so):
    f = Fake()
    W, c, q, s = f(16384 * 2), f(8192), f(256), f(64)
    assert L.call_status("nf4_pack", W, 16384 + 64, c, q, s, None) == L.LM_ERR_SHAPE
    assert L.call_status("nf4_pack", W, 16384, None, q, s, None) == L.LM_ERR_NULL
    assert L.call_status("nf4_pack", W, 16384, W + 32, q, s, None) == L.LM_ERR_ALIAS
    assert L.call_status("nf4_pack", W, 0, c, q, s, None) == L.LM_OK
    assert L.call_status("nf4_dequant", c, q, s, 16384, 9, f(65536), None) == L.LM_ERR_DTYPE
    assert L.call_status("nf4_dequant", c, q, s, 16384, L.LM_OUT_F32, c, None) == L.LM_ERR_ALIAS


def test_int4_argument_errors(so):
    f = Fake()
    W, c, sz = f(256 * 512 * 2), f(256 * 256), f(256 * 512 // 32 * 4)
    assert L.call_status("int4_pack", W, 256, 512, 16, c, sz, None) == L.LM_ERR_SHAPE      # group
    assert L.call_status("int4_pack", W, 256, 96, 64, c, sz, None) == L.LM_ERR_SHAPE       # cols % group
    assert L.call_status("int4_pack", W, 256, 512, 32, None, sz, None) == L.LM_ERR_NULL
    assert L.call_status("int4_pack", W, 256, 512, 32, c, W + 64, None) == L.LM_ERR_ALIAS
    assert L.call_status("int4_pack", W, 0, 512, 128, c, sz, None) == L.LM_OK
    assert L.call_status("int4_dequant", c, sz, 256, 512, 32, 9, f(1 << 20), None) == L.LM_ERR_DTYPE
    assert L.call_status("int4_dequant", c, sz, 256, 512, 32, L.LM_OUT_F32, sz, None) == L.LM_ERR_ALIAS


def test_nvfp4_argument_errors(so):
    f = Fake()
    W, c, sf, gs = f(256 * 512 * 2), f(256 * 256), f(256 * 512 // 16), f(64)
    assert L.call_status("nvfp4_pack", W, 256, 96, c, sf, gs, None) == L.LM_ERR_SHAPE        # cols % 64
    assert L.call_status("nvfp4_pack", W, 256, 512, c, None, gs, None) == L.LM_ERR_NULL
    assert L.call_status("nvfp4_pack", W, 256, 512, c, sf, gs + 2, None) == L.LM_ERR_ALIGN
    assert L.call_status("nvfp4_pack", W, 256, 512, c, sf, W + 64, None) == L.LM_ERR_ALIAS
    assert L.call_status("nvfp4_pack", W, 0, 512, c, sf, gs, None) == L.LM_OK
    assert L.call_status("nvfp4_dequant", c, sf, gs, 256, 512, 9, f(1 << 20), None) == L.LM_ERR_DTYPE
    assert L.call_status("nvfp4_dequant", c, sf, gs, 256, 512, L.LM_OUT_F32, c, None) == L.LM_ERR_ALIAS


def test_nvfp4_weight_validation(so):
    a = _mlp_args()
    for t in ("gate", "up", "down"):
        w = a[t].W
        w.kind, w.codes, w.block_scale, w.global_scale = L.LM_WEIGHT_NVFP4, w.w, w.w + (1 << 24), w.w + (1 << 25)
    a["down"].W.block_scale = None
    assert _fwd(a) == L.LM_ERR_NULL and "down.W.block_scale" in L.last_error()
    a["down"].W.block_scale = a["down"].W.w + (1 << 24)
    a["up"].W.global_scale += 1                                              # a float needs 4-byte alignment
    assert _fwd(a) == L.LM_ERR_ALIGN and "up.W.global_scale" in L.last_error()


def _int4(a, t, group):
    w = a[t].W
    w.kind, w.group = L.LM_WEIGHT_INT4, group
    w.codes = w.w
    w.scale_zero = w.w + (1 << 24)


def test_int4_weight_validation(so):
    # every case fails validation on the host, before any device call
    b = _mlp_args()
    for t in ("gate", "up", "down"):
        _int4(b, t, 64)
    b["up"].W.group = 48
    assert _fwd(b) == L.LM_ERR_SHAPE and "up.W.group" in L.last_error()
    c = _mlp_args()
    for t in ("gate", "up", "down"):
        _int4(c, t, 128)
    c["gate"].W.scale_zero = None
    assert _fwd(c) == L.LM_ERR_NULL and "gate.W.scale_zero" in L.last_error()
    m = _mlp_args()
    _int4(m, "gate", 128)
    assert _fwd(m) == L.LM_ERR_UNSUPPORTED                                   # kinds mixed in one call


def test_profile_summary_empty_without_launches(so):
    L.lm_profile_enable(True)
    L.lm_profile_reset()
    assert L.lm_profile_summary() == {}
    L.lm_profile_enable(False)
    assert L.call_status("lm_profile_summary", None, 0) == L.LM_ERR_NULL


# ---------------------------------------------------------------------------- the other entry points

def _reaches_device(call, a):
    """The untouched argument set passes every host check: without a GPU the call then fails at
    its first CUDA call.  With a GPU present it is not made at all (the fake pointers would be
    launched on)."""
    import torch
    if torch.cuda.is_available():
        return True
    return call(a) in (L.LM_ERR_CUDA, L.LM_ERR_UNSUPPORTED)


def _mlp_bwd_args(T=512, d=256, n=704, r=8):
    a = _mlp_args(T=T, d=d, n=n, r=r)
    f = Fake()
    f.next = 1 << 40
    a.update(dY=f(T * d * 2), dX=f(T * d * 2), dAg=f(r * d * 4), dBg=f(n * r * 4), dAu=f(r * d * 4),
             dBu=f(n * r * 4), dAd=f(r * n * 4), dBd=f(d * r * 4))
    return a


def _bwd(a):
    return L.call_status("lora_mlp_bwd", a["T"], a["d"], a["n"], a["act"], a["X"], a["dY"], a["e"], a["u"], a["h"],
                         a["saved"], a["saved_bytes"], ctypes.byref(a["gate"]), ctypes.byref(a["up"]),
                         ctypes.byref(a["down"]), a["dX"], a["dAg"], a["dBg"], a["dAu"], a["dBu"], a["dAd"],
                         a["dBd"], a["ws"], a["ws_bytes"], None)


def test_mlp_bwd_argument_errors(so):
    a = _mlp_bwd_args()
    assert _reaches_device(_bwd, a)
    assert _bwd(dict(a, dX=None)) == L.LM_ERR_NULL
    assert _bwd(dict(a, dAd=None)) == L.LM_ERR_NULL
    assert _bwd(dict(a, dY=a["dY"] + 2)) == L.LM_ERR_ALIGN
    assert _bwd(dict(a, dX=a["dY"])) == L.LM_ERR_ALIAS                     # output over an input
    assert _bwd(dict(a, dBg=a["dAg"])) == L.LM_ERR_ALIAS                   # two outputs overlap
    assert _bwd(dict(a, ws_bytes=a["ws_bytes"] - 1)) == L.LM_ERR_WORKSPACE
    assert _bwd(dict(a, saved_bytes=16)) == L.LM_ERR_WORKSPACE
    assert _bwd(dict(a, act=7)) == L.LM_ERR_DTYPE
    assert _bwd(dict(a, n=720)) == L.LM_ERR_SHAPE                          # W shapes say 704


def _relu2_args(T=384, d=256, n=512, r=16):
    f = Fake()
    a = dict(T=T, d=d, n=n, X=f(T * d * 2), up=_lora(f, d, n, r), down=_lora(f, n, d, r), y=f(T * d * 2),
             u=f(T * n * 2), h=f(T * n * 2), dY=f(T * d * 2), dX=f(T * d * 2), dAu=f(r * d * 4),
             dBu=f(n * r * 4), dAd=f(r * n * 4), dBd=f(d * r * 4))
    a["saved_bytes"] = _size("lora_relu2_mlp_saved_size", T, r)[1]
    a["saved"] = f(a["saved_bytes"])
    a["ws_bytes"] = _size("lora_relu2_mlp_workspace_size", T, d, n, r)[1]
    a["ws"] = f(a["ws_bytes"])
    return a


def _relu2_fwd(a):
    return L.call_status("lora_relu2_mlp_fwd", a["T"], a["d"], a["n"], a["X"], ctypes.byref(a["up"]),
                         ctypes.byref(a["down"]), a["y"], a["u"], a["h"], a["saved"], a["saved_bytes"], a["ws"],
                         a["ws_bytes"], None)


def _relu2_bwd(a):
    return L.call_status("lora_relu2_mlp_bwd", a["T"], a["d"], a["n"], a["X"], a["dY"], a["u"], a["h"], a["saved"],
                         a["saved_bytes"], ctypes.byref(a["up"]), ctypes.byref(a["down"]), a["dX"], a["dAu"],
                         a["dBu"], a["dAd"], a["dBd"], a["ws"], a["ws_bytes"], None)


def test_relu2_argument_errors(so):
    a = _relu2_args()
    assert _reaches_device(_relu2_fwd, a)
    assert _reaches_device(_relu2_bwd, a)
    assert _relu2_fwd(dict(a, y=None)) == L.LM_ERR_NULL
    assert _relu2_fwd(dict(a, X=a["X"] + 2)) == L.LM_ERR_ALIGN
    assert _relu2_fwd(dict(a, h=a["u"])) == L.LM_ERR_ALIAS
    assert _relu2_fwd(dict(a, ws_bytes=a["ws_bytes"] - 1)) == L.LM_ERR_WORKSPACE
    assert _relu2_fwd(dict(a, d=250)) == L.LM_ERR_SHAPE
    assert _relu2_bwd(dict(a, dBu=None)) == L.LM_ERR_NULL
    assert _relu2_bwd(dict(a, dX=a["X"])) == L.LM_ERR_ALIAS
    assert _relu2_bwd(dict(a, saved_bytes=16)) == L.LM_ERR_WORKSPACE


def _qkv_args(T=300, d=256, nq=256, nk=64, nv=128, r=16):
    f = Fake()
    a = dict(T=T, d=d, nq=nq, nk=nk, nv=nv, X=f(T * d * 2), q=_lora(f, d, nq, r), k=_lora(f, d, nk, r),
             v=_lora(f, d, nv, r), Q=f(T * nq * 2), K=f(T * nk * 2), V=f(T * nv * 2), dQ=f(T * nq * 2),
             dK=f(T * nk * 2), dV=f(T * nv * 2), dX=f(T * d * 2),
             dAq=f(r * d * 4), dBq=f(nq * r * 4), dAk=f(r * d * 4), dBk=f(nk * r * 4), dAv=f(r * d * 4),
             dBv=f(nv * r * 4))
    a["saved_bytes"] = _size("lora_qkv_saved_size", T, r)[1]
    a["saved"] = f(a["saved_bytes"])
    a["ws_bytes"] = _size("lora_qkv_workspace_size", T, d, nq, nk, nv, r)[1]
    a["ws"] = f(a["ws_bytes"])
    return a


def _qkv_fwd(a):
    return L.call_status("lora_qkv_fwd", a["T"], a["d"], a["nq"], a["nk"], a["nv"], a["X"], ctypes.byref(a["q"]),
                         ctypes.byref(a["k"]), ctypes.byref(a["v"]), a["Q"], a["K"], a["V"], a["saved"],
                         a["saved_bytes"], a["ws"], a["ws_bytes"], None)


def _qkv_bwd(a):
    return L.call_status("lora_qkv_bwd", a["T"], a["d"], a["nq"], a["nk"], a["nv"], a["X"], a["dQ"], a["dK"],
                         a["dV"], a["saved"], a["saved_bytes"], ctypes.byref(a["q"]), ctypes.byref(a["k"]),
                         ctypes.byref(a["v"]), a["dX"], a["dAq"], a["dBq"], a["dAk"], a["dBk"], a["dAv"],
                         a["dBv"], a["ws"], a["ws_bytes"], None)


def test_qkv_argument_errors(so):
    a = _qkv_args()                          # K and V of different widths are accepted
    assert _reaches_device(_qkv_fwd, a)
    assert _reaches_device(_qkv_bwd, a)
    assert _qkv_fwd(dict(a, K=None)) == L.LM_ERR_NULL
    assert _qkv_fwd(dict(a, X=a["X"] + 2)) == L.LM_ERR_ALIGN
    assert _qkv_fwd(dict(a, V=a["Q"])) == L.LM_ERR_ALIAS
    assert _qkv_fwd(dict(a, ws_bytes=a["ws_bytes"] - 1)) == L.LM_ERR_WORKSPACE
    assert _qkv_fwd(dict(a, nv=96)) == L.LM_ERR_SHAPE                      # v.W has 128 rows
    b = _qkv_args()
    b["k"].r = 8
    assert _qkv_fwd(b) == L.LM_ERR_SHAPE                                   # ranks differ
    assert _qkv_bwd(dict(a, dBv=None)) == L.LM_ERR_NULL
    assert _qkv_bwd(dict(a, dX=a["dQ"])) == L.LM_ERR_ALIAS
    assert _qkv_bwd(dict(a, saved_bytes=16)) == L.LM_ERR_WORKSPACE


def _o_args(T=257, din=512, dout=256, r=16):
    f = Fake()
    a = dict(T=T, din=din, dout=dout, X=f(T * din * 2), o=_lora(f, din, dout, r), Y=f(T * dout * 2),
             dY=f(T * dout * 2), dX=f(T * din * 2), dA=f(r * din * 4), dB=f(dout * r * 4))
    a["saved_bytes"] = _size("lora_o_saved_size", T, r)[1]
    a["saved"] = f(a["saved_bytes"])
    a["ws_bytes"] = _size("lora_o_workspace_size", T, din, dout, r)[1]
    a["ws"] = f(a["ws_bytes"])
    return a


def _o_fwd(a):
    return L.call_status("lora_o_fwd", a["T"], a["din"], a["dout"], a["X"], ctypes.byref(a["o"]), a["Y"], a["saved"],
                         a["saved_bytes"], a["ws"], a["ws_bytes"], None)


def _o_bwd(a):
    return L.call_status("lora_o_bwd", a["T"], a["din"], a["dout"], a["X"], a["dY"], a["saved"], a["saved_bytes"],
                         ctypes.byref(a["o"]), a["dX"], a["dA"], a["dB"], a["ws"], a["ws_bytes"], None)


def test_o_argument_errors(so):
    a = _o_args()
    assert _reaches_device(_o_fwd, a)
    assert _reaches_device(_o_bwd, a)
    assert _o_fwd(dict(a, Y=None)) == L.LM_ERR_NULL
    assert _o_fwd(dict(a, X=a["X"] + 2)) == L.LM_ERR_ALIGN
    assert _o_fwd(dict(a, Y=a["X"])) == L.LM_ERR_ALIAS
    assert _o_fwd(dict(a, ws_bytes=a["ws_bytes"] - 1)) == L.LM_ERR_WORKSPACE
    assert _o_fwd(dict(a, dout=288)) == L.LM_ERR_SHAPE                     # W has 256 rows
    assert _o_bwd(dict(a, dA=None)) == L.LM_ERR_NULL
    assert _o_bwd(dict(a, dB=a["dA"])) == L.LM_ERR_ALIAS
    assert _o_bwd(dict(a, saved_bytes=16)) == L.LM_ERR_WORKSPACE


def test_empty_token_count_forwards_are_no_ops(so):
    # (the backwards zero their gradients for T = 0, a device call, so they are not made here)
    assert _relu2_fwd(_relu2_args(T=0)) == L.LM_OK
    assert _qkv_fwd(_qkv_args(T=0)) == L.LM_OK
    assert _o_fwd(_o_args(T=0)) == L.LM_OK


def _o_bwd_static(a):
    return L.call_status("lora_o_bwd_static", a["T"], a["din"], a["dout"], a["X"], a["dY"], a["saved"],
                         a["saved_bytes"], ctypes.byref(a["o"]), a["dX"], a["dA"], a["dB"], None)


def test_o_bwd_static_argument_errors_before_any_device_call(so):
    """The static-scratch backward reports every argument error of lora_o_bwd, and a shape too large
    for its scratch, on the host, before it clears the scratch's error word or launches anything."""
    a = _o_args()
    assert _reaches_device(_o_bwd_static, a)
    assert _o_bwd_static(dict(a, dA=None)) == L.LM_ERR_NULL
    assert _o_bwd_static(dict(a, X=a["X"] + 16)) == L.LM_ERR_ALIGN
    assert _o_bwd_static(dict(a, dB=a["dA"])) == L.LM_ERR_ALIAS
    assert _o_bwd_static(dict(a, dX=a["X"])) == L.LM_ERR_ALIAS
    assert _o_bwd_static(dict(a, saved_bytes=16)) == L.LM_ERR_WORKSPACE
    assert _o_bwd_static(dict(a, dout=288)) == L.LM_ERR_SHAPE
    big = _o_args(T=1 << 20, din=4096, dout=4096, r=64)
    assert _o_bwd_static(big) == L.LM_ERR_WORKSPACE
    assert "static scratch" in L.last_error()
