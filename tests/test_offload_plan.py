"""Host logic of the offload decode (skv_offload_plan, no GPU needed): the
batches are runs of whole chunks in order, each within the batch size and
as long as it can be, covering every chunk once."""
import numpy as np
import pytest

from lossless_kv_cache_scalar_gb300 import SKVError
from lossless_kv_cache_scalar_gb300.api import offload_plan


def test_small_cases():
    offs = [0, 16, 32, 48]
    assert offload_plan(offs, 32) == [0, 2, 3]
    assert offload_plan(offs, 48) == [0, 3]
    assert offload_plan(offs, 16) == [0, 1, 2, 3]
    assert offload_plan(offs, 48, max_chunks=2) == [0, 2, 3]  # also capped in chunks
    assert offload_plan([0], 16) == [0]                  # no chunks, no batches
    with pytest.raises(SKVError):
        offload_plan(offs, 15)                           # a chunk larger than a batch
    with pytest.raises(SKVError) as e:
        offload_plan([0, 32, 16, 48], 64)                # descending offsets
    assert e.value.name == "CORRUPT"


@pytest.mark.parametrize("seed", range(5))
def test_random_plans_are_maximal_runs(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 400))
    sizes = 16 * rng.integers(1, 200, n)
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.uint64)
    batch = int(sizes.max() + 16 * rng.integers(0, 600))
    cap = int(rng.integers(0, 20))
    plan = offload_plan(offs, batch, max_chunks=cap)
    assert plan[0] == 0 and plan[-1] == n
    for a, b in zip(plan[:-1], plan[1:]):
        assert b > a and (cap == 0 or b - a <= cap)
        assert int(offs[b] - offs[a]) <= batch
        if b < n:                                        # one more chunk would not fit
            assert int(offs[b + 1] - offs[a]) > batch or b - a == cap
