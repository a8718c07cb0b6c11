"""Failure detection of the tensor-core decode without a GPU fault: the
kernel's waits for its own bulk copies are bounded.  In the library's test
mode (kvq_test_force_stall) each warp's first wait is on a shared-memory
barrier that nothing completes, so the bound runs out for real.  The kernel
must then set KVQ_DEV_STALL, wait (with the normal bound) for the copies it
still has in flight, and return; the context stays usable and the next
normal call gives the normal result."""

import pytest

from tests.gpu_cases import appended_cache

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from bit_kv_cache_04_gb300 import kvq as K  # noqa: E402
from bit_kv_cache_04_gb300 import workloads as W  # noqa: E402


LENGTHS = {"llama2_7b_kivi4": [3000, 1500], "ctx262k_hadamard4": [4000], "mistral7b_hotcold": [6000, 4500]}


@pytest.mark.parametrize("name", sorted(LENGTHS))
def test_wait_that_runs_out_sets_stall_and_returns(name):
    w = W.make(name).scaled(L=2, lengths=LENGTHS[name])
    cache, seq_lens, _, _ = appended_cache(w, with_oracle=False)
    cfg = w.cfg
    q = W.queries(w, cfg.L, "cuda", 3)
    shape = (cfg.L, cfg.batch, cfg.H_q, cfg.D)
    ref = torch.empty(shape, dtype=torch.float32, device="cuda")
    cache.decode(0, cfg.L, q, seq_lens, ref)
    torch.cuda.synchronize()
    assert cache.device_status() == 0
    K.kvq_test_force_stall(256)
    try:
        for splits in (0, 1):
            out = torch.empty(shape, dtype=torch.float32, device="cuda")
            cache.decode(0, cfg.L, q, seq_lens, out, num_splits=splits)
            torch.cuda.synchronize()
            assert cache.device_status() & K.DEV_STALL, splits
            cache.clear_status()
    finally:
        K.kvq_test_force_stall(0)
    torch.cuda.synchronize()
    out = torch.empty(shape, dtype=torch.float32, device="cuda")
    cache.decode(0, cfg.L, q, seq_lens, out)
    torch.cuda.synchronize()
    assert cache.device_status() == 0
    assert torch.equal(out, ref)
