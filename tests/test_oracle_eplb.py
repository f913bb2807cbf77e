"""Pin of the oracle's eplb_local_stats all-gather (CPU only): row r of the
gathered buffer is rank r's statistics, for any element type and rank count
(compared with numpy's stack of the inputs)."""
import numpy as np
import pytest

import oracle


@pytest.mark.parametrize("ep,shape,dtype", [(1, (8,), np.int32), (4, (64,), np.int32),
                                            (32, (8,), np.int64), (64, (3, 4), np.float32)])
def test_gather_is_the_stack_of_ranks(ep, shape, dtype):
    rng = np.random.default_rng(ep)
    local = [rng.integers(-1000, 1000, size=shape).astype(dtype) for _ in range(ep)]
    got = oracle.eplb_gather(local)
    want = np.stack(local).reshape(ep, -1).view(np.uint8).reshape(ep, -1)
    np.testing.assert_array_equal(got, want)
    # a rank's row does not depend on the others
    local2 = [x.copy() for x in local]
    local2[ep // 2] = local2[ep // 2] + np.ones(shape, dtype)
    got2 = oracle.eplb_gather(local2)
    same = [r for r in range(ep) if r != ep // 2]
    np.testing.assert_array_equal(got2[same], got[same])
