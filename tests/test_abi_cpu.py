"""Host-side checks of the C ABI that need no GPU: the library builds, loads and exports
every declared entry point; sizes and argument checks answer without touching CUDA."""

import ctypes
import os
import re

import pytest

from post_weight_quantization_02_gb300 import gptq as G

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(gptq_\w+)\s*\(", src))
    return sorted(names)


def test_library_exports_every_declared_symbol():
    lib = G.lib()
    names = declared_functions()
    assert "gptq_hessian_accumulate" in names and len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    assert G.gptq_abi_version() == 1


def test_status_names():
    assert G.gptq_status_string(G.GPTQ_ERR_NOT_PD) == "GPTQ_ERR_NOT_PD"
    assert G.gptq_kernel_name(0) == "syrk_tc"


def test_workspace_sizes():
    d, m = 4096, 4096
    assert G.gptq_workspace_size(G.GPTQ_OP_PREPARE, 0, 0, d) >= 2 * d * d * 4
    q = G.gptq_workspace_size(G.GPTQ_OP_QUANTIZE, 0, m, d, 4, 128)
    assert q >= m * d * 5 + 128 * m * 4
    h = G.gptq_workspace_size(G.GPTQ_OP_HESSIAN, 262144, 0, d)
    assert h >= d * d * 4 + 256
    assert G.gptq_workspace_size(G.GPTQ_OP_QUANTIZE, 0, m, d, 4, 96) == 0
    assert G.gptq_workspace_size(9, 0, m, d, 4, 128) == 0


# Fake, aligned, never-dereferenced addresses: every call below fails its argument
# checks before anything reaches CUDA.
P = 1 << 20


def _call_q(**kw):
    a = dict(W=P, wdtype=1, U=P, perm=None, dead=None, m=64, d=256, bits=4, group=128, sym=0,
             block=128, qw=P, sc=P, qz=P, gi=P, loss=P, ws=P, wsb=1 << 30)
    a.update(kw)
    return G.lib().gptq_quantize_layer(a["W"], a["wdtype"], a["U"], a["perm"], a["dead"],
                                       a["m"], a["d"], a["bits"], a["group"], a["sym"],
                                       a["block"], a["qw"], a["sc"], a["qz"], a["gi"],
                                       a["loss"], a["ws"], a["wsb"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(bits=5), G.GPTQ_ERR_UNSUPPORTED),
    (dict(group=96), G.GPTQ_ERR_UNSUPPORTED),
    (dict(group=128, block=96), G.GPTQ_ERR_UNSUPPORTED),
    (dict(d=250), G.GPTQ_ERR_UNSUPPORTED),
    (dict(m=48), G.GPTQ_ERR_UNSUPPORTED),
    (dict(U=None), G.GPTQ_ERR_INVALID_ARG),
    (dict(block=0), G.GPTQ_ERR_INVALID_ARG),
    (dict(sym=2), G.GPTQ_ERR_INVALID_ARG),
    (dict(wdtype=7), G.GPTQ_ERR_INVALID_ARG),
    (dict(W=P + 4), G.GPTQ_ERR_INVALID_ARG),
    (dict(m=-1), G.GPTQ_ERR_INVALID_ARG),
    (dict(wsb=1024), G.GPTQ_ERR_WORKSPACE),
])
def test_quantize_argument_checks(kw, status):
    assert _call_q(**kw) == status
    assert G.gptq_last_error() != ""


def test_prepare_and_hessian_argument_checks():
    lib = G.lib()
    info = ctypes.c_int32(-5)
    assert lib.gptq_prepare(P, 0, 0.01, 1, P, P, P, ctypes.byref(info), P, 1 << 30, None) \
        == G.GPTQ_ERR_INVALID_ARG
    assert info.value == 0
    assert lib.gptq_prepare(P, 100, 0.01, 1, P, P, P, None, P, 1 << 30, None) == \
        G.GPTQ_ERR_UNSUPPORTED
    assert lib.gptq_prepare(P, 128, -1.0, 1, P, P, P, None, P, 1 << 30, None) == \
        G.GPTQ_ERR_INVALID_ARG
    assert lib.gptq_prepare(P, 128, 0.01, 1, P, P, P, None, P, 1000, None) == \
        G.GPTQ_ERR_WORKSPACE
    n = ctypes.c_int64(0)
    assert lib.gptq_hessian_accumulate(P, ctypes.byref(n), P, 3, 10, 128, P, 1 << 30, None) \
        == G.GPTQ_ERR_INVALID_ARG
    assert lib.gptq_hessian_accumulate(P, ctypes.byref(n), P, 1, 10, 100, P, 1 << 30, None) \
        == G.GPTQ_ERR_UNSUPPORTED
    assert lib.gptq_hessian_accumulate(P, ctypes.byref(n), P, 1, 10, 128, P, 100, None) \
        == G.GPTQ_ERR_WORKSPACE
    assert lib.gptq_hessian_accumulate(None, ctypes.byref(n), P, 1, 10, 128, P, 1 << 30, None) \
        == G.GPTQ_ERR_INVALID_ARG
    assert n.value == 0


def _call_dq(**kw):
    a = dict(x=P, xt=1, n=4, d=256, m=64, bits=4, qw=P, sc=P, qz=P, gi=P, G=2, y=P, ws=P,
             wsb=256)
    a.update(kw)
    return G.lib().gptq_dequant_matmul(a["x"], a["xt"], a["n"], a["d"], a["m"], a["bits"],
                                       a["qw"], a["sc"], a["qz"], a["gi"], a["G"], a["y"],
                                       a["ws"], a["wsb"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(bits=5), G.GPTQ_ERR_UNSUPPORTED),
    (dict(d=250), G.GPTQ_ERR_UNSUPPORTED),
    (dict(m=48), G.GPTQ_ERR_UNSUPPORTED),
    (dict(xt=9), G.GPTQ_ERR_INVALID_ARG),
    (dict(G=0), G.GPTQ_ERR_INVALID_ARG),
    (dict(n=-1), G.GPTQ_ERR_INVALID_ARG),
    (dict(ws=P + 4), G.GPTQ_ERR_INVALID_ARG),
    (dict(wsb=8), G.GPTQ_ERR_INVALID_ARG),
    (dict(y=None), G.GPTQ_ERR_INVALID_ARG),
    (dict(qw=P + 4), G.GPTQ_ERR_INVALID_ARG),   # copied 16 bytes at a time
    (dict(sc=P + 8), G.GPTQ_ERR_INVALID_ARG),
])
def test_dequant_matmul_argument_checks(kw, status):
    assert _call_dq(**kw) == status


def test_quantize_flags_and_dequant_workspace():
    assert G.gptq_workspace_size(G.GPTQ_OP_DEQUANT_MATMUL, 0, 64, 256, 4, -1) >= 256
    # an unknown quantize flag is rejected before anything reaches CUDA
    assert G.lib().gptq_quantize_layer_ex(P, 1, P, None, None, 64, 256, 4, 128, 0, 128, 2, P,
                                          P, P, P, P, P, 1 << 30, None) == \
        G.GPTQ_ERR_INVALID_ARG


def _call_host(**kw):
    a = dict(X=P, xt=1, ntok=4096, chunk=1024, W=P, wt=1, m=64, d=256, damp=0.01, act=1,
             bits=4, group=128, sym=0, block=128, flags=0, qw=P, sc=P, qz=P, gi=P, perm=P,
             dev=P, devb=1 << 40)
    a.update(kw)
    loss = ctypes.c_double(0.0)
    info = ctypes.c_int32(0)
    return G.lib().gptq_quantize_layer_host(
        a["X"], a["xt"], a["ntok"], a["chunk"], a["W"], a["wt"], a["m"], a["d"], a["damp"],
        a["act"], a["bits"], a["group"], a["sym"], a["block"], a["flags"], a["qw"], a["sc"],
        a["qz"], a["gi"], a["perm"], ctypes.byref(loss), ctypes.byref(info), a["dev"],
        a["devb"], None)


@pytest.mark.parametrize("kw,status,msg", [
    (dict(ntok=0, X=None), G.GPTQ_ERR_INVALID_ARG, "no calibration tokens"),
    (dict(W=None), G.GPTQ_ERR_INVALID_ARG, "null"),
    (dict(chunk=0), G.GPTQ_ERR_INVALID_ARG, "chunk_tokens"),
    (dict(xt=7), G.GPTQ_ERR_INVALID_ARG, "dtypes"),
    (dict(damp=-1.0), G.GPTQ_ERR_INVALID_ARG, "damp"),
    (dict(flags=4), G.GPTQ_ERR_INVALID_ARG, "flags"),
    (dict(bits=5), G.GPTQ_ERR_UNSUPPORTED, "bits"),
    (dict(group=96), G.GPTQ_ERR_UNSUPPORTED, "group"),
    (dict(group=256, block=96), G.GPTQ_ERR_UNSUPPORTED, "divide"),
    (dict(m=48), G.GPTQ_ERR_UNSUPPORTED, "multiples of 32"),
    (dict(dev=P + 16), G.GPTQ_ERR_INVALID_ARG, "256-byte aligned"),
    (dict(devb=4096), G.GPTQ_ERR_WORKSPACE, "too small"),
])
def test_layer_host_argument_checks(kw, status, msg):
    """gptq_quantize_layer_host rejects bad arguments before any copy or kernel."""
    assert _call_host(**kw) == status
    assert msg in G.gptq_last_error()


def test_layer_host_size_and_the_other_additions():
    lib = G.lib()
    n = G.gptq_layer_host_size(16384, 8192, 28672, 4, 128, G.GPTQ_BF16, G.GPTQ_BF16)
    # at least H, U, two staging chunks and W, and the largest of the three scratch uses
    assert n >= 2 * 28672 ** 2 * 4 + 2 * 16384 * 28672 * 2 + 8192 * 28672 * 2 + \
        G.gptq_workspace_size(G.GPTQ_OP_PREPARE, 0, 0, 28672)
    assert G.gptq_layer_host_size(16384, 8192, 28672, 4, 128, G.GPTQ_F32, G.GPTQ_BF16) > n
    assert G.gptq_layer_host_size(0, 64, 256, 4, 128, 1, 1) == 0
    assert G.gptq_layer_host_size(1024, 64, 250, 4, 128, 1, 1) == 0
    assert G.gptq_layer_host_size(1024, 64, 256, 5, 128, 1, 1) == 0
    # gptq_hessian_rescale and gptq_check_wait_timeout check their arguments first
    assert lib.gptq_hessian_rescale(None, 256, 1, 2, None) == G.GPTQ_ERR_INVALID_ARG
    assert lib.gptq_hessian_rescale(P, 256, 1, 0, None) == G.GPTQ_ERR_INVALID_ARG
    assert lib.gptq_hessian_rescale(P, 256, -1, 2, None) == G.GPTQ_ERR_INVALID_ARG
    assert lib.gptq_hessian_rescale(P, 100, 1, 2, None) == G.GPTQ_ERR_UNSUPPORTED
    assert lib.gptq_hessian_rescale(P + 4, 256, 1, 2, None) == G.GPTQ_ERR_INVALID_ARG
    assert lib.gptq_check_wait_timeout(0, P, 256, None) == G.GPTQ_ERR_INVALID_ARG
    assert lib.gptq_check_wait_timeout(2 * 10 ** 9, P, 256, None) == G.GPTQ_ERR_INVALID_ARG
    assert lib.gptq_check_wait_timeout(1000, P + 8, 256, None) == G.GPTQ_ERR_INVALID_ARG
    assert lib.gptq_check_wait_timeout(1000, P, 16, None) == G.GPTQ_ERR_INVALID_ARG
    # the fp16 scale copy checks its arguments before any launch; n = 0 does nothing
    assert lib.gptq_scales_fp16(P, -1, P, None) == G.GPTQ_ERR_INVALID_ARG
    assert lib.gptq_scales_fp16(None, 8, P, None) == G.GPTQ_ERR_INVALID_ARG
    assert lib.gptq_scales_fp16(P, 8, None, None) == G.GPTQ_ERR_INVALID_ARG
    assert lib.gptq_scales_fp16(None, 0, None, None) == G.GPTQ_OK
    # the SYRK's wait limit: 0 (the default) or 1 .. 1e10 ns, a host-side setting
    assert lib.gptq_set_wait_limit(2 * 10 ** 10) == G.GPTQ_ERR_INVALID_ARG
    assert lib.gptq_set_wait_limit(5) == G.GPTQ_OK
    assert lib.gptq_set_wait_limit(0) == G.GPTQ_OK
