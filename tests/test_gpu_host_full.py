"""The host-buffer call (gptq_quantize_layer_host) at the 70B-width down_proj's full size:
524,288 bf16 tokens in page-locked host memory (30.5 GB), copied in 16,384-token chunks
beside the Hessian kernels, then W, then the packed outputs back.  Its outputs equal, bit
for bit, those of the device path fed the same chunks (the same Hessian recurrence, so the
same Hessian, permutation and factor); the device path's outputs are checked against the
float64 oracle at this size in the large tests."""

import pytest
import torch

from post_weight_quantization_02_gb300 import LayerEngine, quantize_layer_from_host
from workloads import CONFIGS, channel_multipliers, make_tokens_chunk, make_weight

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def test_host_call_full_size_matches_device_path(lib, cuda_device):
    cfg = CONFIGS["down_proj_8192x28672"]
    dev = cuda_device
    m, d, n, ch = cfg.d_out, cfg.d_in, cfg.n_tokens, cfg.chunk
    mult = channel_multipliers(cfg, dev)
    eng_dev = LayerEngine(m, d, cfg.bits, cfg.group, cfg.sym, cfg.actorder, cfg.damp,
                          cfg.blocksize, max_chunk_tokens=ch, device=dev)
    Xh = torch.empty(n, d, dtype=cfg.x_dtype, pin_memory=True)
    for i, t0 in enumerate(range(0, n, ch)):
        X = make_tokens_chunk(cfg, i, dev, mult)
        eng_dev.add_batch(X)
        Xh[t0:t0 + ch].copy_(X)
        del X
    W = make_weight(cfg, dev)
    res_dev = eng_dev.quantize(W).to("cpu")
    torch.cuda.synchronize()
    Wh = W.cpu().pin_memory()
    del W, eng_dev
    torch.cuda.empty_cache()
    eng = LayerEngine(m, d, cfg.bits, cfg.group, cfg.sym, cfg.actorder, cfg.damp,
                      cfg.blocksize, max_chunk_tokens=ch, device=dev)
    res_host = quantize_layer_from_host(eng, Wh, Xh, chunk_tokens=ch)
    for f in ("qweight", "scales", "qzeros", "g_idx", "perm", "loss"):
        assert torch.equal(getattr(res_host, f), getattr(res_dev, f)), f
