"""The allocation-free decode attention (``kivi_decode_attention_noalloc``):
its split workspace is the library's fixed device array.  Two consecutive
calls must give exactly what the workspace-taking entry point gives on the
same cache (same kernels, same split count, so the same bits).  Collected
last so that nothing else runs after a call that used the shared array."""
from __future__ import annotations

import math

import numpy as np
import pytest

import workloads as W
from gpu_util import to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU-only machines
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import kv_cache_quantization_kivi_gb300 as K  # noqa: E402


def test_noalloc_matches_workspace_entry_point():
    layers, batch, h_kv, r, d = 2, 2, 4, 4, 128
    bh = batch * h_kv
    cache = K.KiviCache(layers, bh, d, r_cap=128, cap=512, group=32, bits=2, residual=32)
    w = W.custom(seed=71, batch=1, kv_heads=bh, seq=600, head_dim=d)
    pos = 0
    for n in (70, 60, 64, 50, 64, 40, 60, 44):
        for l in range(layers):
            cache.append(l, to_dev(W.generate(w, l, "k", tok0=pos, n_tok=n)),
                         to_dev(W.generate(w, l, "v", tok0=pos, n_tok=n)))
        cache.advance(n)
        pos += n
        cache.flush()
    assert cache.s_q >= 256 and cache.n_res > 0
    rng = np.random.default_rng(5)
    q = torch.from_numpy(rng.standard_normal((layers, batch, h_kv * r, d)).astype(np.float16)).cuda()
    sc = 1.0 / math.sqrt(d)
    for n_split in (1, 3):
        ref = cache.decode_attention(q, batch, sm_scale=sc, n_split=n_split)
        outs = []
        for _ in range(2):
            out = torch.full((layers, batch, h_kv * r, d), float("nan"), device="cuda")
            K.kivi_decode_attention_noalloc(cache.layers, layers, cache.state, batch, h_kv * r,
                                            sc, list(q.unbind(0)), list(out.unbind(0)), n_split)
            outs.append(out)
        torch.cuda.synchronize()
        assert K.kivi_device_fault() == 0
        for out in outs:
            assert torch.equal(out, ref), n_split
