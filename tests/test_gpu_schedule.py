"""The device tile scheduler is integer work: bit-exact against the oracle's
schedule rule on every workload and on random length mixes (zeros included)."""
import numpy as np
import pytest
import torch

from variable_length_flashattention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vfa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from variable_length_flashattention_gb300 import build, vfa as binding
    build.build()
    return binding


def _check(vfa, oracle_mod, lq, lk, H, bq, bk, causal, pair=False, window_left=-1):
    cq, ck = W.cu_seqlens(lq), W.cu_seqlens(lk)
    items, status = vfa.schedule(torch.from_numpy(cq).cuda(), torch.from_numpy(ck).cuda(),
                                 int(cq[-1]), int(ck[-1]), max(lq), H, bq, bk, causal, pair,
                                 window_left=window_left)
    assert status == 0
    ref = oracle_mod.schedule(cq, ck, H, bq, bk, causal, pair, window_left=window_left)
    got = items.cpu().numpy()
    assert got.shape == ref.shape
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("name", ["tiny", "tiny-causal", "packed", "longtail", "cross-d64",
                                  "cross-d256"])
def test_workload_schedules(vfa, oracle_mod, name):
    case = W.VARLEN_WORKLOADS[name](0)
    bq, bk, pair = vfa.tile_shape(case.head_dim)
    _check(vfa, oracle_mod, case.lengths_q, case.lengths_k, case.num_heads, bq, bk, case.causal,
           pair)


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("causal", [False, True, 2])
def test_random_mixes(vfa, oracle_mod, seed, causal):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 3000 if seed == 5 else 60))
    lq = [int(x) for x in rng.integers(0, 1500, B)]
    lk = [int(x) for x in rng.integers(0, 1500, B)]
    lq[0] = max(lq[0], 1)
    for bq, bk in ((128, 128), (128, 64)):
        for pair in (False, True):
            _check(vfa, oracle_mod, lq, lk, int(rng.integers(1, 5)), bq, bk, causal, pair)


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("causal", [1, 2])
def test_window_random_mixes(vfa, oracle_mod, seed, causal):
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 3000 if seed == 3 else 60))
    lq = [int(x) for x in rng.integers(0, 3000, B)]
    lk = [int(x) for x in rng.integers(0, 3000, B)]
    lq[0] = max(lq[0], 1)
    for window_left in (0, 1, 100, 128, 1000, int(rng.integers(0, 5000)), 1 << 30):
        for bq, bk in ((128, 128), (128, 64)):
            for pair in (False, True):
                _check(vfa, oracle_mod, lq, lk, int(rng.integers(1, 4)), bq, bk, causal, pair,
                       window_left)


def test_many_tiles_use_global_scratch(vfa, oracle_mod):
    # more than 4096 q tiles and 4096 cost buckets: the scheduler's global-memory path
    lq = [128] * 4200 + [700000]
    lk = [1] * 4200 + [700000]
    _check(vfa, oracle_mod, lq, lk, 1, 128, 128, True)
    _check(vfa, oracle_mod, lq, lk, 1, 128, 128, True, pair=True)
    _check(vfa, oracle_mod, lq, lk, 1, 128, 128, True, pair=True, window_left=5000)


def test_bad_seqlens_status(vfa):
    cu = torch.tensor([0, 5, 3, 9], dtype=torch.int32, device="cuda")
    items, status = vfa.schedule(cu, cu, 9, 9, 9, 1, 128, 128, True)
    assert status == vfa.VFA_ERR_BAD_SEQLENS and items.shape[0] == 0
