"""hs_pool_touch_host: the GPU reads the whole host pool once and changes
nothing (host rows byte-identical afterwards, no device error)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import sparse_attention_kv_hs_gb300 as hs  # noqa: E402


@pytest.mark.parametrize("kv_format", [0, 1])
def test_touch_host_reads_the_pool_and_changes_nothing(kv_format):
    pool = hs.Pool(2, 3, 256, 512, 256, 576, 8, 5000, 4, kv_format)
    rng = np.random.default_rng(7 + kv_format)
    pool.host_pool[...] = rng.integers(0, 1 << 16, size=pool.host_pool.shape, dtype=np.uint16)
    before = pool.host_pool.copy()
    s = torch.cuda.Stream()
    hs.hs_pool_touch_host(pool.handle, s)
    s.synchronize()
    assert np.array_equal(pool.host_pool, before)
    assert hs.hs_check_errors(pool.handle) == 0
    pool.close()
