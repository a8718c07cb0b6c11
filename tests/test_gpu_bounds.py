"""The bounds-checked build (libkvq_checked.so, compiled with
KVQ_BOUNDS_CHECK) stands in for a memory checker: every computed cache
address is checked against its buffer segment (layer, sequence, kv head, row
or page), and a miss sets KVQ_DEV_BOUNDS and skips the access.

* On every kernel path (per-channel and per-token appends, the tiers'
  requantization, the window ring, paged rotated and per-token rows, the tensor-core and
  generic decodes, the fused decode step, dequantize), across the tiny-shape
  sweep's lengths and scaled workloads, no check fires and the bytes still
  equal the oracle's.
* With the test hook that treats each segment's last row as outside it,
  the checks fire (and the run stays clean: the skipped accesses never
  leave the buffers)."""

import json
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCALED = {
    "llama2_7b_kivi4": dict(L=2, lengths=[700, 333, 129]),
    "mistral7b_hotcold": dict(L=1, lengths=[4500, 4390, 200]),
    "gqa8b_hadamard4_paged": dict(L=2, lengths=[300, 77, 129, 16]),
    "ctx262k_hadamard3": dict(L=1, lengths=[777]),
    "ctx262k_tbq4": dict(L=1, lengths=[400]),
    "q4_0_mha_1k": dict(L=1, lengths=[1000]),
    "llama2_7b_kivi2_zp": dict(L=1, lengths=[500, 64]),
}


def _checked_run():
    """Runs in a fresh interpreter with KVQ_LIBRARY pointing at the checked
    build; prints one JSON line of per-case results."""
    sys.path.insert(0, ROOT)
    from bit_kv_cache_04_gb300 import kvq as K
    from bit_kv_cache_04_gb300 import workloads as W
    from tests.gpu_cases import PAGED_PER_TOKEN, appended_cache, gpu_buffers_as_oracle, paged_workload
    from tests.helpers import oracle_cfg
    from tests.test_gpu_tiny_shapes import CASES as TINY, LENGTHS as TINY_LENGTHS, _cfg as tiny_cfg

    assert K.LIB_PATH.endswith("libkvq_checked.so"), K.LIB_PATH
    res = {}

    def exercise(name, w):
        cfg = w.cfg
        cache, seq_lens, ref, table = appended_cache(w, chunks=[97, 1, 33, 256])
        got = gpu_buffers_as_oracle(cache, oracle_cfg(cfg))
        same = all(np.array_equal(got[n], ref[n]) for n in ref)
        q = W.queries(w, cfg.L, "cuda", 3)
        out = torch.empty((cfg.L, cfg.batch, cfg.H_q, cfg.D), dtype=torch.float32, device="cuda")
        cache.decode(0, cfg.L, q, seq_lens, out)
        for splits in (1, 3):
            cache.decode(0, cfg.L, q, seq_lens, out, num_splits=splits)
        gen = torch.Generator().manual_seed(5)
        dt = torch.float16 if cfg.in_dtype == K.DT_F16 else torch.bfloat16
        cu1 = torch.arange(0, cfg.batch + 1, dtype=torch.int32, device="cuda")
        for _ in range(3):
            kn = torch.randn((cfg.L, cfg.batch, cfg.H_kv, cfg.D), generator=gen).to(dt).cuda()
            vn = torch.randn((cfg.L, cfg.batch, cfg.H_kv, cfg.D), generator=gen).to(dt).cuda()
            cache.decode_step(0, cfg.L, kn, vn, q, seq_lens, out)
            cache.commit_lengths(cu1, seq_lens)
        T = int(seq_lens[0].item())
        kd = torch.empty((max(T, 1), cfg.H_kv, cfg.D), dtype=torch.float32, device="cuda")
        cache.dequantize(0, 0, 0, T, seq_lens, kd[:T], torch.empty_like(kd)[:T])
        torch.cuda.synchronize()
        res[name] = {"status": cache.device_status(), "bytes_equal": bool(same),
                     "finite": bool(torch.isfinite(out).all())}

    for name, kw in SCALED.items():
        exercise(name, W.make(name).scaled(**kw))
    for key in PAGED_PER_TOKEN:
        exercise(key, paged_workload(key))
    for kind, D, R in TINY:
        cfg, values = tiny_cfg(kind, D, R)
        exercise(f"tiny_{kind}_d{D}_r{R}", W.Workload(f"tiny_{kind}", cfg, list(TINY_LENGTHS), values, 40))

    # the hook: every segment's last row counts as outside it
    K.kvq_test_shrink_bounds(1)
    try:
        # the 16-bit window ring (160 slots) wraps at 400 tokens, so its last slot is used
        w = W.make("llama2_7b_kivi4").scaled(L=1, lengths=[400, 64], extra=0)
        cache, seq_lens, _, _ = appended_cache(w, with_oracle=False)
        q = W.queries(w, 1, "cuda", 3)
        out = torch.empty((1, w.cfg.batch, w.cfg.H_q, w.cfg.D), dtype=torch.float32, device="cuda")
        cache.decode(0, 1, q, seq_lens, out)
        torch.cuda.synchronize()
        res["shrunk"] = {"status": cache.device_status()}
    finally:
        K.kvq_test_shrink_bounds(0)
    print(json.dumps(res))


@pytest.fixture(scope="module")
def checked_results():
    sys.path.insert(0, ROOT)
    from bit_kv_cache_04_gb300 import _build

    lib = _build.build(checked=True)
    env = dict(os.environ, KVQ_LIBRARY=lib)
    r = subprocess.run([sys.executable, "-c", "import tests.test_gpu_bounds as t; t._checked_run()"],
                       capture_output=True, text=True, env=env, cwd=ROOT, timeout=1800)
    assert r.returncode == 0, r.stderr[-4000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_no_check_fires_on_any_kernel_path(checked_results):
    from bit_kv_cache_04_gb300 import kvq as K

    for name, r in checked_results.items():
        if name == "shrunk":
            continue
        assert r["status"] == 0, (name, r)
        assert r["bytes_equal"] and r["finite"], (name, r)


def test_checks_fire_when_segments_are_shrunk(checked_results):
    from bit_kv_cache_04_gb300 import kvq as K

    assert checked_results["shrunk"]["status"] & K.DEV_BOUNDS
