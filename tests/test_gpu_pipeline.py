"""The whole layer path on the GPU (Hessian -> prepare -> quantize) against the oracle run
on the same inputs from scratch."""

import numpy as np
import pytest
import torch

from oracle import gptq_oracle as O
from post_weight_quantization_02_gb300 import LayerEngine, quantize_layer_from_host
from tests.parity import check_quantize, to_np
from workloads import CONFIGS, make_weight, token_chunks

pytestmark = pytest.mark.gpu


def _outputs(res):
    return dict(qweight=to_np(res.qweight), scales=to_np(res.scales), qzeros=to_np(res.qzeros),
                g_idx=to_np(res.g_idx), loss=float(res.loss))


@pytest.mark.parametrize("name,override", [
    ("layer_256x256", {}),
    ("layer_256x256", dict(x_dtype=torch.bfloat16, w_dtype=torch.bfloat16, actorder=True,
                           group=64, bits=3, sym=True)),
])
def test_layer_end_to_end(lib, cuda_device, name, override):
    cfg = CONFIGS[name].replace(**override)
    eng = LayerEngine(cfg.d_out, cfg.d_in, cfg.bits, cfg.group, cfg.sym, cfg.actorder, cfg.damp,
                      cfg.blocksize, max_chunk_tokens=cfg.chunk, device=cuda_device)
    chunks = list(token_chunks(cfg))
    for X in chunks:
        eng.add_batch(X.to(cuda_device))
    W = make_weight(cfg)
    res = eng.quantize(W.to(cuda_device))
    torch.cuda.synchronize()
    X = torch.cat(chunks).float().numpy()
    ref = O.gptq_prepare(O.hessian(X), cfg.damp, cfg.actorder)
    assert np.array_equal(to_np(res.perm), ref["perm"])
    check_quantize(W.float().numpy().astype(np.float64), ref["U"], ref["perm"], ref["dead"],
                   cfg.bits, cfg.group, cfg.sym, _outputs(res))


def test_layer_from_host_matches_device_path(lib, cuda_device):
    """The host-buffer call (gptq_quantize_layer_host: chunked copies overlapped with the
    Hessian kernels) gives the device path's outputs bit for bit with the same chunking."""
    cfg = CONFIGS["layer_256x256"].replace(chunk=512)
    chunks = list(token_chunks(cfg))
    X = torch.cat(chunks).pin_memory()
    W = make_weight(cfg).pin_memory()
    eng = LayerEngine(cfg.d_out, cfg.d_in, cfg.bits, cfg.group, cfg.sym, cfg.actorder, cfg.damp,
                      max_chunk_tokens=cfg.chunk, device=cuda_device)
    host = quantize_layer_from_host(eng, W, X, chunk_tokens=cfg.chunk)
    eng2 = LayerEngine(cfg.d_out, cfg.d_in, cfg.bits, cfg.group, cfg.sym, cfg.actorder, cfg.damp,
                       max_chunk_tokens=cfg.chunk, device=cuda_device)
    for c in chunks:
        eng2.add_batch(c.to(cuda_device))
    dev = eng2.quantize(W.to(cuda_device)).to("cpu")
    for f in ("qweight", "scales", "qzeros", "g_idx", "perm", "loss"):
        assert torch.equal(getattr(host, f), getattr(dev, f)), f
    # a second call on the same buffers gives the same outputs; a ragged last chunk (300
    # tokens per chunk) matches the device path fed the same chunks
    again = quantize_layer_from_host(eng, W, X, chunk_tokens=cfg.chunk)
    for f in ("qweight", "scales", "qzeros", "g_idx", "perm", "loss"):
        assert torch.equal(getattr(again, f), getattr(dev, f)), f
    ragged = quantize_layer_from_host(eng, W, X, chunk_tokens=300)
    eng3 = LayerEngine(cfg.d_out, cfg.d_in, cfg.bits, cfg.group, cfg.sym, cfg.actorder, cfg.damp,
                       max_chunk_tokens=300, device=cuda_device)
    for t0 in range(0, X.shape[0], 300):
        eng3.add_batch(X[t0:t0 + 300].to(cuda_device))
    dev3 = eng3.quantize(W.to(cuda_device)).to("cpu")
    for f in ("qweight", "scales", "qzeros", "g_idx", "perm", "loss"):
        assert torch.equal(getattr(ragged, f), getattr(dev3, f)), f


def test_layer_from_host_rejects_empty_tokens(lib, cuda_device):
    cfg = CONFIGS["layer_256x256"]
    eng = LayerEngine(cfg.d_out, cfg.d_in, cfg.bits, cfg.group, cfg.sym, cfg.actorder, cfg.damp,
                      device=cuda_device)
    with pytest.raises(lib.GptqError, match="no calibration tokens"):
        quantize_layer_from_host(eng, make_weight(cfg), torch.empty(0, cfg.d_in))
