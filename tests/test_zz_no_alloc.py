"""kvq_decode_attention_static: decode attention for callers that cannot
allocate device memory (no workspace argument; the library keeps its scratch
in a fixed device array).

Through the C ABI, two calls in a row must give the output of
kvq_decode_attention on the same cache, within the tolerance the tests use
between two GPU decode paths.  This file is collected last and also passes
alone in a fresh process.
"""

import ctypes

import numpy as np
import pytest

from tests.gpu_cases import appended_cache
from tests.helpers import rel_err

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from bit_kv_cache_04_gb300 import kvq as K  # noqa: E402
from bit_kv_cache_04_gb300 import workloads as W  # noqa: E402

TOL_GPU_PATHS = 1e-5

CASES = {
    # 16-bit window, split partials in the scratch
    "llama2_7b_kivi4": (dict(L=2, lengths=[700, 333, 129]), 0),
    # RoPE tables in the scratch
    "mistral7b_hotcold": (dict(L=1, lengths=[4500, 200]), 0),
    # explicit split count
    "gqa8b_hadamard4_paged": (dict(L=2, lengths=[300, 77, 129, 16]), 7),
}


def _static_call(cache, n_layers, q, seq_lens, out, splits):
    return K.LIB.kvq_decode_attention_static(ctypes.byref(cache.c_cfg), ctypes.byref(cache.c_cache), 0, n_layers,
                                             q.data_ptr(), seq_lens.data_ptr(), out.data_ptr(), splits,
                                             torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("name", sorted(CASES))
def test_static_scratch_matches_workspace_path(name):
    kw, splits = CASES[name]
    w = W.make(name).scaled(**kw)
    cfg = w.cfg
    cache, seq_lens, _, _ = appended_cache(w, with_oracle=False)
    q = W.queries(w, cfg.L, "cuda", seed=3)
    shape = (cfg.L, cfg.batch, cfg.H_q, cfg.D)
    ref = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
    cache.decode(0, cfg.L, q, seq_lens, ref, num_splits=splits)
    torch.cuda.synchronize()
    ref = ref.cpu().numpy()
    assert np.isfinite(ref).all()
    for _ in range(2):
        out = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
        st = _static_call(cache, cfg.L, q, seq_lens, out, splits)
        assert st == 0, K.LIB.kvq_last_error().decode()
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert np.isfinite(got).all()
        assert rel_err(got, ref) <= TOL_GPU_PATHS


def test_static_scratch_rejects_oversized_call():
    cfg = K.Config(L=4, H_kv=8, H_q=32, D=128, batch=64, max_T=4096, k_fmt=K.Fmt(4, 32, K.AXIS_CHANNEL),
                   v_fmt=K.Fmt(4, 32), residual_window=128)
    cache = K.KVCache(cfg, "cuda")
    q = torch.zeros((4, 64, 32, 128), dtype=torch.float16, device="cuda")
    out = torch.zeros((4, 64, 32, 128), dtype=torch.float32, device="cuda")
    sl = torch.zeros(64, dtype=torch.int32, device="cuda")
    st = _static_call(cache, 4, q, sl, out, 256)
    assert st == 5  # KVQ_ERR_WORKSPACE
    assert "static scratch" in K.LIB.kvq_last_error().decode()
    torch.cuda.synchronize()
    assert torch.all(out == 0)
