"""Tiny-shape sweep against the CPU oracle: every sequence length around the
32-token tile and group edges (0, 1, 15, 16, 17, 31, 33, 127, 129 tokens, one
sequence each, in one ragged batch) x head dim 128 / 256 x no window / a
128-token window, for per-channel KIVI blocks, per-token blocks, rotated
128-value blocks and hot/cold tiers with pre-RoPE keys.  Each case checks:

* the packed cache is byte-identical to the oracle's;
* decode attention is within 2e-3 of fp64 attention over the same bytes
  (an empty sequence gives 0);
* one fused decode step (one new token per sequence) leaves the oracle's
  bytes and attends to the grown cache within the same bound;
* no device status bit is set.
"""

import numpy as np
import pytest

from oracle import kvq_oracle as O
from tests.gpu_cases import appended_cache, gpu_buffers_as_oracle
from tests.helpers import oracle_cfg, raw16, rel_err

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from bit_kv_cache_04_gb300 import kvq as K  # noqa: E402
from bit_kv_cache_04_gb300 import workloads as W  # noqa: E402

LENGTHS = [0, 1, 15, 16, 17, 31, 33, 127, 129]
TOL = 2e-3


def _cfg(kind, D, R):
    dt = K.DT_F16 if D == 128 else K.DT_BF16
    base = dict(L=2, H_kv=2, H_q=4, D=D, batch=len(LENGTHS), max_T=max(LENGTHS) + 40, in_dtype=dt,
                residual_window=R)
    if kind == "kivi4":
        return K.Config(k_fmt=K.Fmt(4, 32, K.AXIS_CHANNEL), v_fmt=K.Fmt(4, 32), **base), "mha_1k"
    if kind == "token4":
        return K.Config(k_fmt=K.Fmt(4, 32), v_fmt=K.Fmt(4, 32), **base), "mha_1k"
    if kind == "rot4_128":
        return K.Config(k_fmt=K.Fmt(4, 128), v_fmt=K.Fmt(4, 128), flags=K.ROTATE_K | K.ROTATE_V,
                        sign_seed=W.SIGN_SEED, **base), "mha_1k"
    if kind == "hotcold_rope":
        base["in_dtype"] = K.DT_F16
        return K.Config(k_fmt=K.Fmt(4, 32, K.AXIS_CHANNEL), v_fmt=K.Fmt(4, 32), k_cold=K.Fmt(2, 32, K.AXIS_CHANNEL),
                        v_cold=K.Fmt(2, 32), hot_window=64, flags=K.K_PRE_ROPE, rope_theta=10000.0,
                        **base), "mistral"
    raise KeyError(kind)


CASES = [(k, D, R) for k in ("kivi4", "token4", "rot4_128", "hotcold_rope") for D in (128, 256) for R in (0, 128)]


@pytest.mark.parametrize("case", CASES, ids=[f"{k}-d{D}-r{R}" for k, D, R in CASES])
def test_tiny_shapes_against_oracle(case):
    kind, D, R = case
    cfg, values = _cfg(kind, D, R)
    w = W.Workload(f"tiny_{kind}", cfg, list(LENGTHS), values, 40)
    cache, seq_lens, ref, table = appended_cache(w)
    oc = oracle_cfg(cfg)
    got = gpu_buffers_as_oracle(cache, oc)
    assert cache.device_status() == 0
    for n in ref:
        assert np.array_equal(got[n], ref[n]), (case, n)
    q = W.queries(w, cfg.L, "cuda", 5)
    out = torch.full((cfg.L, cfg.batch, cfg.H_q, D), float("nan"), dtype=torch.float32, device="cuda")
    cache.decode(0, cfg.L, q, seq_lens, out)
    torch.cuda.synchronize()
    o_ref = O.decode_attention(oc, got, 0, cfg.L, raw16(q), LENGTHS, block_table=table)
    assert torch.isfinite(out).all()
    assert rel_err(out.cpu().numpy(), o_ref) <= TOL, case
    assert torch.all(out[:, 0] == 0)  # the empty sequence attends to nothing
    # one fused decode step: the new token appended, attention over T + 1 tokens
    gen = torch.Generator().manual_seed(11)
    dt = torch.float16 if cfg.in_dtype == K.DT_F16 else torch.bfloat16
    kn = torch.randn((cfg.L, cfg.batch, cfg.H_kv, D), generator=gen).to(dt)
    vn = torch.randn((cfg.L, cfg.batch, cfg.H_kv, D), generator=gen).to(dt)
    q1 = W.queries(w, cfg.L, "cuda", 6)
    cache.decode_step(0, cfg.L, kn.cuda(), vn.cuda(), q1, seq_lens, out)
    torch.cuda.synchronize()
    assert cache.device_status() == 0
    for l in range(cfg.L):
        O.append(oc, ref, l, raw16(kn[l]), raw16(vn[l]), [1] * cfg.batch, LENGTHS, block_table=table)
    got = gpu_buffers_as_oracle(cache, oc)
    for n in ref:
        assert np.array_equal(got[n], ref[n]), (case, "step", n)
    o_ref = O.decode_attention(oc, got, 0, cfg.L, raw16(q1), [t + 1 for t in LENGTHS], block_table=table)
    assert rel_err(out.cpu().numpy(), o_ref) <= TOL, (case, "step")
