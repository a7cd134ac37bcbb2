"""The Python binding's own checks, on the CPU: buffer element types and sizes are
checked before anything reaches the library, and well-formed calls (the patterns the GPU
tests use, empty layers included) pass through with the arguments in the ABI's order.

The ctypes library is replaced by a recorder and CPU tensors stand in for device
buffers, so nothing here needs a GPU or runs a kernel."""

import pytest
import torch

from post_weight_quantization_02_gb300 import gptq as G


class _Recorder:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def call(*args):
            self.calls.append((name, args))
            return 256 if name == "gptq_workspace_size" else G.GPTQ_OK
        return call


@pytest.fixture
def rec(monkeypatch):
    r = _Recorder()
    monkeypatch.setattr(G, "lib", lambda: r)
    # CPU tensors stand in for device buffers: their address is the "pointer"
    monkeypatch.setattr(G, "_ptr", lambda t: None if t is None else t.data_ptr())
    monkeypatch.setattr(G, "_stream", lambda s: 0)
    return r


def _layer(m=64, d=256, bits=4, group=128):
    G_ = 1 if group == -1 else -(-d // group)
    return dict(W=torch.zeros(m, d), U=torch.eye(d), perm=torch.arange(d, dtype=torch.int32),
                dead=torch.zeros(d, dtype=torch.uint8),
                qweight=torch.zeros(bits * d // 32, m, dtype=torch.int32),
                scales=torch.zeros(G_, m), qzeros=torch.zeros(G_, bits * m // 32, dtype=torch.int32),
                g_idx=torch.zeros(d, dtype=torch.int32), loss=torch.zeros((), dtype=torch.float64))


def _quantize(L, bits=4, group=128, **over):
    L = dict(L, **over)
    G.gptq_quantize_layer(L["W"], L["U"], L["perm"], L["dead"], bits, group, False, 128,
                          L["qweight"], L["scales"], L["qzeros"], L["g_idx"], L["loss"],
                          ws=torch.zeros(256, dtype=torch.uint8))


def test_quantize_well_formed(rec):
    L = _layer()
    _quantize(L)
    name, args = rec.calls[-1]
    assert name == "gptq_quantize_layer_ex"
    assert args[2] == L["U"].data_ptr() and args[3] == L["perm"].data_ptr()
    assert args[12] == L["qweight"].data_ptr() and args[16] == L["loss"].data_ptr()
    _quantize(L, perm=None, dead=None)                       # optional buffers
    L3 = _layer(m=96, d=384, bits=3, group=-1)
    _quantize(L3, bits=3, group=-1)


def test_quantize_empty_layer(rec):
    """Zero rows: flat empty outputs are accepted (their sizes are all zero)."""
    d = 128
    empty = torch.empty(0, dtype=torch.int32)
    G.gptq_quantize_layer(torch.empty(0, d), torch.eye(d), None, None, 4, 128, False, 128,
                          empty, empty.float(), empty, torch.zeros(d, dtype=torch.int32),
                          torch.zeros((), dtype=torch.float64),
                          ws=torch.zeros(256, dtype=torch.uint8))
    assert rec.calls[-1][0] == "gptq_quantize_layer_ex"


@pytest.mark.parametrize("field,bad,msg", [
    ("perm", torch.arange(256, dtype=torch.int64), "perm must be torch.int32"),
    ("dead", torch.zeros(256, dtype=torch.bool), "dead must be torch.uint8"),
    ("U", torch.eye(256, dtype=torch.float64), "Hinv_chol must be torch.float32"),
    ("g_idx", torch.zeros(255, dtype=torch.int32), "g_idx must hold 256"),
    ("scales", torch.zeros(1, 64), "scales must hold 128"),
    ("qweight", torch.zeros(16, 64, dtype=torch.int32), "qweight must hold 2048"),
    ("qzeros", torch.zeros(2, 8, dtype=torch.int64), "qzeros must be torch.int32"),
    ("loss", torch.zeros((), dtype=torch.float32), "loss must be torch.float64"),
])
def test_quantize_bad_buffer(rec, field, bad, msg):
    with pytest.raises(ValueError, match=msg):
        _quantize(_layer(), **{field: bad})
    assert not any(c[0] == "gptq_quantize_layer_ex" for c in rec.calls)


def test_quantize_sizes_left_to_the_library(rec):
    """Invalid bits or group sizes are the library's to reject (with its own status)."""
    L = _layer()
    _quantize(L, bits=5)
    _quantize(L, group=0)
    assert [c[0] for c in rec.calls].count("gptq_quantize_layer_ex") == 2


def test_prepare_and_hessian(rec):
    d = 64
    H, U = torch.eye(d), torch.zeros(d, d)
    perm, dead = torch.zeros(d, dtype=torch.int32), torch.zeros(d, dtype=torch.uint8)
    ws = torch.zeros(256, dtype=torch.uint8)
    assert G.gptq_prepare(H, 0.01, True, perm, dead, U, ws) == 0
    with pytest.raises(ValueError, match="perm must be torch.int32"):
        G.gptq_prepare(H, 0.01, True, perm.long(), dead, U, ws)
    with pytest.raises(ValueError, match="H must be torch.float32"):
        G.gptq_prepare(H.double(), 0.01, True, perm, dead, U, ws)
    X = torch.zeros(8, d, dtype=torch.bfloat16)
    G.gptq_hessian_accumulate(H, 0, X, ws)
    G.gptq_hessian_accumulate_async(H, 0, X, ws)
    with pytest.raises(ValueError, match="H must be torch.float32"):
        G.gptq_hessian_accumulate(H.half(), 0, X, ws)


def _checkpoint(m=64, d=256, bits=4, G_=2):
    return (torch.zeros(bits * d // 32, m, dtype=torch.int32), torch.zeros(G_, m),
            torch.zeros(G_, bits * m // 32, dtype=torch.int32), torch.zeros(d, dtype=torch.int32))


def test_dequant_well_formed_and_checked(rec):
    qw, sc, qz, gi = _checkpoint()
    ws = torch.zeros(256, dtype=torch.uint8)
    y = G.gptq_dequant_matmul(torch.zeros(3, 256, dtype=torch.bfloat16), qw, sc, qz, gi, 4, ws=ws)
    assert y.shape == (3, 64)
    name, args = rec.calls[-1]
    assert name == "gptq_dequant_matmul"
    assert args[6:10] == (qw.data_ptr(), sc.data_ptr(), qz.data_ptr(), gi.data_ptr())
    assert args[10] == 2 and args[11] == y.data_ptr()
    W = G.gptq_dequantize(qw, sc, qz, gi, 4, dtype=torch.float32, ws=ws)
    assert W.shape == (64, 256)
    with pytest.raises(ValueError, match="qweight must hold"):
        G.gptq_dequant_matmul(torch.zeros(3, 512, dtype=torch.bfloat16), qw, sc, qz, gi, 4, ws=ws)
    with pytest.raises(ValueError, match="g_idx must be torch.int32"):
        G.gptq_dequant_matmul(torch.zeros(3, 256), qw, sc, qz, gi.long(), 4, ws=ws)
    with pytest.raises(ValueError, match="y must hold"):
        G.gptq_dequant_matmul(torch.zeros(3, 256), qw, sc, qz, gi, 4, y=torch.zeros(2, 64), ws=ws)
    with pytest.raises(ValueError, match="W must hold"):
        G.gptq_dequantize(qw, sc, qz, gi, 4, W=torch.zeros(64, 255), ws=ws)
