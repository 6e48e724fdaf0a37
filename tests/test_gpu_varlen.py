"""GPU parity of vfa_varlen_fwd against the fp64 oracle (through the C ABI).

Every workload (tiny, packed, long-tail, cross-attention at D=64 and D=256)
at seeds 0, 1 and 2, compared element by element over every output row, in
the launch configuration the bench times; the long-tail workload (32768
tokens, H=32, about a minute of oracle time per seed on 16 cores) too.
Edge cases and variants on smaller shapes.  Outputs start as NaN canaries,
so a row the kernel never wrote fails.
"""
import numpy as np
import pytest
import torch

from helpers import FLT_MAX, assert_lse_close, assert_out_close, run_varlen, to_dev
from variable_length_flashattention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vfa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from variable_length_flashattention_gb300 import build, vfa as binding
    build.build()
    return binding


def _oracle_full(oracle_mod, case):
    out, lse, _ = oracle_mod.varlen_fwd(case.q, case.k, case.v, case.cu_seqlens_q,
                                        case.cu_seqlens_k, case.num_heads, case.head_dim,
                                        case.softmax_scale, case.causal)
    return out, lse


def _check_full(vfa, oracle_mod, case):
    out, lse, status = run_varlen(vfa, case)
    assert status == 0, f"device status {status}"
    ref_out, ref_lse = _oracle_full(oracle_mod, case)
    assert_out_close(out, ref_out, case.name)
    assert_lse_close(lse, ref_lse, case.name)


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("causal", [False, True])
def test_tiny(vfa, oracle_mod, causal, seed):
    _check_full(vfa, oracle_mod, W.tiny(causal, seed))


@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_row_counts_at_warp_boundaries(vfa, oracle_mod, head_dim, causal):
    # The pair kernel writes a tile's output 32 rows (one warp) at a time: by a
    # tile store when all 32 rows belong to the sequence, by plain stores of
    # the existing rows otherwise (rows past the sequence are the next
    # sequence's).  Lengths at, just below and just above multiples of 32 and
    # of the 128-row tile put every warp of a tile on both sides of that
    # boundary, with the next sequence's rows right behind.
    lengths = [31, 32, 33, 63, 64, 65, 96, 127, 128, 129, 160, 191, 224, 255, 256, 257]
    case = W.make_varlen("warp-rows", lengths, lengths, 2, head_dim, causal, 1.0,
                         value_seed=head_dim + 3 * causal)
    _check_full(vfa, oracle_mod, case)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_packed_training_batch(vfa, oracle_mod, seed):
    _check_full(vfa, oracle_mod, W.packed(seed))


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("head_dim", [64, 256])
def test_cross_attention(vfa, oracle_mod, head_dim, seed):
    case = W.cross(head_dim, seed)
    assert sum(1 for x in case.lengths_k if x == 1) >= 4
    _check_full(vfa, oracle_mod, case)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_longtail_full(vfa, oracle_mod, seed):
    # all 32768 x 32 (token, head) rows against the oracle, compared in slices
    # of tokens to bound the host memory the comparison takes
    case = W.longtail(seed)
    assert case.total_q == 32768 and max(case.lengths_q) == 8192
    out, lse, status = run_varlen(vfa, case)
    assert status == 0
    ref_out, ref_lse = _oracle_full(oracle_mod, case)
    for t0 in range(0, case.total_q, 4096):
        t1 = min(case.total_q, t0 + 4096)
        assert_out_close(out[t0:t1], ref_out[t0:t1], f"longtail seed {seed} tokens {t0}..")
        assert_lse_close(lse[t0:t1], ref_lse[t0:t1], f"longtail seed {seed} tokens {t0}..")


EDGE = [
    # (lengths_q, lengths_k, H, D, causal)
    ([0, 5, 0, 130], [3, 0, 0, 130], 2, 128, False),       # empty q rows, empty key sets
    ([0, 5, 0, 130], [3, 0, 0, 130], 2, 128, True),
    ([1, 127, 128, 129, 256, 257], [1, 127, 128, 129, 256, 257], 3, 64, True),
    ([1, 127, 128, 129, 256, 257], [1, 127, 128, 129, 256, 257], 3, 256, True),
    ([300, 7, 1], [40, 300, 1], 2, 128, True),             # Lq > Lk and Lq < Lk, top-left causal
    ([300, 7, 1], [40, 300, 1], 2, 256, True),
    ([200, 64], [65, 500], 1, 256, False),
    ([1] * 40, [1] * 40, 4, 64, True),                       # many one-token sequences
]


@pytest.mark.parametrize("lq,lk,H,D,causal", EDGE)
def test_edge_shapes(vfa, oracle_mod, lq, lk, H, D, causal):
    case = W.make_varlen("edge", lq, lk, H, D, causal, 1.0, value_seed=sum(lq) + D)
    _check_full(vfa, oracle_mod, case)


def test_large_logits_rescale_path(vfa, oracle_mod):
    # sigma 3: scaled logits span tens of units, so the running max jumps by more
    # than the lazy-rescale threshold many times along a row
    case = W.make_varlen("wide", [700, 300], [700, 900], 2, 128, True, 3.0, value_seed=9)
    # V at the workloads' scale (sigma 1): the tolerance is stated for outputs of that size
    case.v = W.bf16_normal(tuple(case.v.shape), 1.0, torch.Generator().manual_seed(10))
    _check_full(vfa, oracle_mod, case)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_rising_scores_rescale_every_tile(vfa, oracle_mod, D, causal):
    # q . k grows by more than 2^8 (in log2 units) every 64 keys along each
    # sequence: every key tile after the first moves the reference max, so the
    # kernel rescales O and l at every tile (after waiting for the previous
    # tile's O += P V) and the D = 256 kernel, whose tiles are 64 keys, at
    # every tile too.
    lengths = [700, 300, 64, 129]
    case = W.make_varlen("rising", lengths, lengths, 2, D, causal, 0.3, value_seed=D + 7)
    q = case.q.float()
    k = case.k.float()
    q[:, :, 0] = 4.0
    cq = case.cu_seqlens_q
    for b in range(len(lengths)):
        pos = torch.arange(lengths[b], dtype=torch.float32)
        k[int(cq[b]):int(cq[b + 1]), :, 0] = (0.5 * pos)[:, None]
    case.q = q.to(torch.bfloat16)
    case.k = k.to(torch.bfloat16)
    case.v = W.bf16_normal(tuple(case.v.shape), 1.0, torch.Generator().manual_seed(D))
    _check_full(vfa, oracle_mod, case)


@pytest.mark.parametrize("H,Hkv,D", [(8, 2, 128), (8, 1, 64), (4, 2, 256), (16, 4, 128)])
@pytest.mark.parametrize("causal", [False, True])
def test_grouped_kv_heads(vfa, oracle_mod, H, Hkv, D, causal):
    # K/V with fewer heads than Q: query head h reads kv head h // (H // Hkv)
    lq, lk = [300, 7, 129, 0, 64, 1], [300, 40, 129, 5, 200, 1]
    case = W.make_varlen("gqa", lq, lk, H, D, causal, 1.0, value_seed=10 * H + Hkv + D)
    case.k = case.k[:, :Hkv].contiguous()
    case.v = case.v[:, :Hkv].contiguous()
    out, lse, status = run_varlen(vfa, case)
    assert status == 0
    ref_out, ref_lse, _ = oracle_mod.varlen_fwd(case.q, case.k, case.v, case.cu_seqlens_q,
                                                case.cu_seqlens_k, H, D, case.softmax_scale,
                                                causal, num_kv_heads=Hkv)
    assert_out_close(out, ref_out, f"gqa {H}/{Hkv}/{D}")
    assert_lse_close(lse, ref_lse, f"gqa {H}/{Hkv}/{D}")


@pytest.mark.parametrize("D", [64, 128, 256])
def test_bottom_right_causal(vfa, oracle_mod, D):
    # causal == 2: local key j visible to local query i iff j <= i + Lk - Lq
    # (chunked-prefill shape: a query block at the end of a longer key sequence,
    # and the reverse, where the first rows see no key at all)
    lq = [64, 300, 129, 500, 1, 0, 200]
    lk = [1000, 300, 40, 128, 77, 5, 0]
    case = W.make_varlen("bottom-right", lq, lk, 2, D, True, 1.0, value_seed=D + 3)
    case.causal = 2
    out, lse, status = run_varlen(vfa, case)
    assert status == 0
    ref_out, ref_lse, _ = oracle_mod.varlen_fwd(case.q, case.k, case.v, case.cu_seqlens_q,
                                                case.cu_seqlens_k, 2, D, case.softmax_scale, 2)
    assert_out_close(out, ref_out, f"bottom-right D={D}")
    assert_lse_close(lse, ref_lse, f"bottom-right D={D}")


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [1, 2])
@pytest.mark.parametrize("window_left", [0, 37, 128, 300])
def test_sliding_window(vfa, oracle_mod, D, causal, window_left):
    # keys j with i + off - window_left <= j <= i + off; ragged lengths, Lq > Lk
    # (rows past the keys' end see nothing) and Lq < Lk both ways
    lq = [64, 700, 129, 500, 1, 0, 260, 1000]
    lk = [1000, 700, 40, 128, 77, 5, 0, 600]
    case = W.make_varlen("window", lq, lk, 2, D, True, 1.0, value_seed=D + window_left)
    case.causal = causal
    out, lse, status = run_varlen(vfa, case, window_left=window_left)
    assert status == 0
    ref_out, ref_lse, _ = oracle_mod.varlen_fwd(case.q, case.k, case.v, case.cu_seqlens_q,
                                                case.cu_seqlens_k, 2, D, case.softmax_scale,
                                                causal, window_left=window_left)
    what = f"window {window_left} causal {causal} D={D}"
    assert_out_close(out, ref_out, what)
    assert_lse_close(lse, ref_lse, what)


def test_sliding_window_grouped_kv_heads(vfa, oracle_mod):
    lq, lk = [300, 1, 900, 77], [300, 50, 900, 500]
    case = W.make_varlen("window-gqa", lq, lk, 8, 128, True, 1.0, value_seed=5)
    case.k = case.k[:, :2].contiguous()
    case.v = case.v[:, :2].contiguous()
    out, lse, status = run_varlen(vfa, case, window_left=200)
    assert status == 0
    ref_out, ref_lse, _ = oracle_mod.varlen_fwd(case.q, case.k, case.v, case.cu_seqlens_q,
                                                case.cu_seqlens_k, 8, 128, case.softmax_scale,
                                                True, num_kv_heads=2, window_left=200)
    assert_out_close(out, ref_out, "window gqa")
    assert_lse_close(lse, ref_lse, "window gqa")


@pytest.mark.parametrize("window_left", [1000, 4095])
def test_sliding_window_long_sequence_sampled(vfa, oracle_mod, window_left):
    case = W.make_varlen("long-window", [16384], [16384], 1, 128, True, 1.0, value_seed=6)
    out, lse, status = run_varlen(vfa, case, window_left=window_left)
    assert status == 0
    rows = np.stack([np.r_[0:64, 8000:8064, 16320:16384], np.zeros(192, int)], 1).astype(np.int64)
    ref_out, ref_lse, _ = oracle_mod.varlen_fwd_rows(case.q, case.k, case.v, case.cu_seqlens_q,
                                                     case.cu_seqlens_k, 1, 128,
                                                     case.softmax_scale, True, rows,
                                                     window_left=window_left)
    assert_out_close(out[rows[:, 0], rows[:, 1]], ref_out, "long window")
    assert_lse_close(lse[rows[:, 0], rows[:, 1]], ref_lse, "long window")


def test_single_long_sequence_sampled(vfa, oracle_mod):
    case = W.make_varlen("long", [16384], [16384], 1, 128, True, 1.0, value_seed=4)
    out, lse, status = run_varlen(vfa, case)
    assert status == 0
    rows = np.stack([np.r_[0:64, 8000:8064, 16320:16384], np.zeros(192, int)], 1).astype(np.int64)
    ref_out, ref_lse, _ = oracle_mod.varlen_fwd_rows(case.q, case.k, case.v, case.cu_seqlens_q,
                                                     case.cu_seqlens_k, 1, 128,
                                                     case.softmax_scale, True, rows)
    assert_out_close(out[rows[:, 0], rows[:, 1]], ref_out, "long")
    assert_lse_close(lse[rows[:, 0], rows[:, 1]], ref_lse, "long")


def test_deterministic(vfa):
    case = W.packed(2)
    a = run_varlen(vfa, case)
    b = run_varlen(vfa, case)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


@pytest.mark.parametrize("bad", ["start", "decreasing", "end", "max_seqlen"])
def test_bad_cu_seqlens_sets_status_and_writes_nothing(vfa, bad):
    case = W.tiny(True, 0)
    d = to_dev(case)
    cu_q = d["cu_q"].clone()
    max_q = case.max_seqlen_q
    if bad == "start":
        cu_q[0] = 1
    elif bad == "decreasing":
        cu_q[2] = cu_q[1] - 1
    elif bad == "end":
        cu_q[-1] = cu_q[-1] - 1
    else:
        max_q = 100
    out = torch.full_like(d["q"], 7.0)
    lse = torch.full((case.total_q, 2), 7.0, device="cuda")
    ws = vfa.alloc_workspace(case.batch, case.total_q, case.total_k, 2, 64)
    vfa.varlen_fwd(d["q"], d["k"], d["v"], cu_q, d["cu_k"], max_q, case.softmax_scale, True,
                   out=out, lse=lse, workspace=ws)
    assert vfa.read_status(ws) == vfa.VFA_ERR_BAD_SEQLENS
    assert torch.all(out == 7.0) and torch.all(lse == 7.0)
    # the same workspace is usable again afterwards
    out2, lse2, status = run_varlen(vfa, case, workspace=ws)
    assert status == 0 and np.all(np.isfinite(out2))


def test_scale_and_plan_example(vfa):
    # the plan's two-independent-sequences example, through the GPU path
    H, D = 1, 64
    cu = torch.tensor([0, 3, 7], dtype=torch.int32, device="cuda")
    vals = torch.tensor([1.0] * 3 + [100.0] * 4)[:, None, None].expand(-1, H, D)
    x = vals.contiguous().to(torch.bfloat16).cuda()
    out, lse = vfa.varlen_fwd(x, x, x, cu, cu, 4, 0.5, False)
    o = out.float().cpu()
    assert torch.allclose(o[:3], torch.ones(3, H, D)) and torch.allclose(o[3:], torch.full((4, H, D), 100.0))
