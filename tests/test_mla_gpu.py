"""GPU parity of MLA decode attention with weight absorption
(b200q_mla_absorb) against the CPU oracle qref_mla_absorb, element by element,
within 1e-5 of the oracle's bound; and the paged-cache append."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import TOL_F32, assert_within, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import torch
    torch.cuda.set_device(0)
    import quantized_weight_quant_gb300 as q
    return q


def _case(fmt, H, Dn, Dv, K, R, S, T, seed, gs=0):
    codes, sc = synth.quant_tensor(fmt, H * (Dn + Dv), K, seed, 1, 5e-3, 2e-2)
    if gs:
        sc = synth.uniform_f32((H * (Dn + Dv), -(-K // gs)), 5e-3, 2e-2, seed, 6)
    qn = synth.normal_f32((S, H, Dn), seed, 2, std=4.0)
    qr = synth.normal_f32((S, H, R), seed, 3)
    lat = synth.normal_f32((T, K), seed, 4)
    rope = synth.normal_f32((T, R), seed, 5)
    return codes, sc, qn, qr, lat, rope


def _run(q, fmt, H, Dn, Dv, K, R, S, T, st0, scale, seed=0, order=None, garbage=True, gs=0):
    """Caches filled through b200q_kv_append into pages placed by `order`;
    with `garbage`, positions before st0 and the rest of the last page
    (positions >= T) hold NaN."""
    import torch
    codes, sc, qn, qr, lat, rope = _case(fmt, H, Dn, Dv, K, R, S, T, seed, gs)
    if garbage:                    # rows before the window: NaN, which neither side may read
        lat[:st0] = np.nan
        rope[:st0] = np.nan
    n_pages = -(-T // 64)
    if order == "reversed":
        order = list(range(n_pages))[::-1]
    kv = q.PagedKV(K, R, T, order=order)
    if garbage:
        kv.lat_pool.fill_(float("nan"))
        kv.rope_pool.fill_(float("nan"))
    kv.append(to_dev(lat), to_dev(rope) if R else None, 0, T)
    ctx = torch.empty((S, H, Dv), dtype=torch.float32, device="cuda")
    with q.tensor_upload(fmt, H * (Dn + Dv), K, codes, sc, gs=gs) as t:
        kv.attend(t, H, Dn, Dv, to_dev(qn), to_dev(qr) if R else None, T, st0, scale, ctx, S)
        torch.cuda.synchronize()
        assert q.device_status() == q.OK
        got = ctx.cpu().numpy()
    ref, bound = oracle.mla_absorb(fmt, H, Dn, Dv, K, codes, sc, qn, qr, lat, rope, st0, scale, gs=gs)
    return got, ref, bound


SMALL = [  # fmt, H, Dn, Dv, K, R, S, T, st0
    (0, 3, 8, 5, 40, 8, 1, 70, 0),
    (1, 2, 16, 12, 64, 4, 3, 130, 5),
    (2, 5, 7, 9, 132, 12, 2, 33, 31),
    (3, 4, 12, 6, 96, 8, 4, 200, 0),
    (2, 1, 4, 4, 16, 0, 1, 1, 0),          # one position, no rope
    (2, 6, 32, 32, 256, 32, 5, 64, 59),    # st0 = T - S
    (1, 17, 8, 8, 48, 4, 1, 97, 40),       # H * S not a multiple of 16
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "f%d_H%d_K%d_R%d_S%d_T%d_st%d" % (c[0], c[1], c[4], c[5], c[6], c[7], c[8]))
@pytest.mark.parametrize("order", [None, "reversed"], ids=["pages_in_order", "pages_reversed"])
def test_mla_small_vs_oracle(q, case, order):
    fmt, H, Dn, Dv, K, R, S, T, st0 = case
    got, ref, bound = _run(q, fmt, H, Dn, Dv, K, R, S, T, st0, 0.35, seed=H + T, order=order)
    assert_within(got.reshape(S, -1), ref.reshape(S, -1), bound.reshape(S, -1), TOL_F32, str(case))


@pytest.mark.parametrize("S", [1, 4])
def test_mla_full_size_int4(q, S):
    """64 heads, nope / value 128, latent 512, rope 64, 4096 cached positions."""
    H, Dn, Dv, K, R, T = 64, 128, 128, 512, 64, 4096
    got, ref, bound = _run(q, 2, H, Dn, Dv, K, R, S, T, 0, (Dn + R) ** -0.5, seed=7, garbage=False)
    assert_within(got.reshape(S, -1), ref.reshape(S, -1), bound.reshape(S, -1), TOL_F32, "full S=%d" % S)


@pytest.mark.parametrize("T,st0", [(20000, 0), (20000, 19000), (5000, 1234)])
def test_mla_long_cache_sampled_heads(q, T, st0):
    """Long caches (many tiles per split, windows that start mid-page): all
    outputs against the oracle run on a few heads of the same tensor."""
    H, Dn, Dv, K, R, S = 16, 64, 64, 256, 32, 2
    got, ref, bound = _run(q, 2, H, Dn, Dv, K, R, S, T, st0, 0.1, seed=T + st0, garbage=False)
    assert_within(got.reshape(S, -1), ref.reshape(S, -1), bound.reshape(S, -1), TOL_F32, "T=%d" % T)


def test_mla_peaked_scores(q):
    """Large scores (one position dominates each softmax): the running max and
    the split combine must not overflow or lose it."""
    got, ref, bound = _run(q, 1, 4, 16, 16, 64, 8, 2, 300, 0, 8.0, seed=3)
    assert np.all(np.isfinite(got))
    assert_within(got.reshape(2, -1), ref.reshape(2, -1), bound.reshape(2, -1), TOL_F32, "peaked")


def test_kv_append_places_rows(q):
    import torch
    K, R, T = 12, 4, 150
    kv = q.PagedKV(K, R, T, order=[2, 0, 1])
    lat = synth.normal_f32((T, K), 1, 1)
    rope = synth.normal_f32((T, R), 1, 2)
    kv.append(to_dev(lat[:100]), to_dev(rope[:100]), 0, 100)      # in two calls, the second mid-page
    kv.append(to_dev(lat[100:]), to_dev(rope[100:]), 100, T - 100)
    torch.cuda.synchronize()
    pool_l, pool_r = kv.lat_pool.cpu().numpy(), kv.rope_pool.cpu().numpy()
    for pos in range(T):
        slot = kv.slots[pos // 64]
        assert np.array_equal(pool_l[slot, pos % 64], lat[pos])
        assert np.array_equal(pool_r[slot, pos % 64], rope[pos])


def test_mla_bad_page_is_reported(q):
    """A NULL page inside the window is never read; the call reports it through
    b200q_device_status and the context stays usable."""
    import torch
    H, Dn, Dv, K, R, S, T = 2, 4, 4, 16, 4, 1, 130
    codes, sc, qn, qr, lat, rope = _case(2, H, Dn, Dv, K, R, S, T, 5)
    kv = q.PagedKV(K, R, T)
    kv.append(to_dev(lat), to_dev(rope), 0, T)
    kv.lat_pages[1] = 0
    ctx = torch.empty((S, H, Dv), dtype=torch.float32, device="cuda")
    with q.tensor_upload(2, H * (Dn + Dv), K, codes, sc) as t:
        kv.attend(t, H, Dn, Dv, to_dev(qn), to_dev(qr), T, 0, 0.5, ctx, S)
        with pytest.raises(q.B200QError) as ei:
            q.device_status()
        assert ei.value.status == q.EINVAL and "page" in str(ei.value)
        assert q.device_status() == q.OK               # the record was cleared
        kv.attend(t, H, Dn, Dv, to_dev(qn), to_dev(qr), T, 128, 0.5, ctx, S)   # page 1 outside the window
        torch.cuda.synchronize()
        assert q.device_status() == q.OK


def test_mla_argument_errors(q):
    import torch
    H, Dn, Dv, K, R = 2, 4, 4, 16, 4
    codes, sc = synth.quant_tensor(2, H * (Dn + Dv), K, 0, 1, 5e-3, 2e-2)
    kv = q.PagedKV(K, R, 64)
    qn = torch.zeros((1, H, Dn), device="cuda")
    qr = torch.zeros((1, H, R), device="cuda")
    ctx = torch.empty((1, H, Dv), device="cuda")
    with q.tensor_upload(2, H * (Dn + Dv), K, codes, sc) as t:
        for args, what in [((3, Dn, Dv), "rows"), ((H, Dn, Dv + 1), "rows")]:
            with pytest.raises(q.B200QError) as ei:
                kv.attend(t, *args, qn, qr, 10, 0, 0.5, ctx, 1)
            assert ei.value.status == q.EINVAL
        with pytest.raises(q.B200QError):
            kv.attend(t, H, Dn, Dv, qn, qr, 10, 10, 0.5, ctx, 1)          # st0 > T - S
        with pytest.raises(q.B200QError):
            kv.attend(t, H, Dn, Dv, qn, qr, 0, 0, 0.5, ctx, 1)            # T < S
        with pytest.raises(q.B200QError):
            kv.attend(t, H, Dn, Dv, qn, qr, 10, 0, float("nan"), ctx, 1)
        with pytest.raises(q.B200QError):
            kv.attend(t, H, Dn, Dv, qn, qr, 10, 0, 0.5, qn, 1)           # ctx overlaps q_nope
        kv.attend(t, H, Dn, Dv, qn, qr, 10, 0, 0.5, ctx, 0)              # S = 0: no-op
    c6, s6 = synth.quant_tensor(2, H * (Dn + Dv), 18, 0, 1, 5e-3, 2e-2)
    with q.tensor_upload(2, H * (Dn + Dv), 18, c6, s6) as t:
        kv18 = q.PagedKV(18, R, 64)
        with pytest.raises(q.B200QError):
            kv18.attend(t, H, Dn, Dv, qn, qr, 10, 0, 0.5, ctx, 1)        # K not a multiple of 4


GS_CASES = [  # fmt, gs, H, Dn, Dv, K, R, S, T, st0
    (2, 32, 3, 16, 12, 256, 8, 2, 150, 3), (2, 128, 4, 8, 8, 512, 16, 1, 100, 0), (2, 16, 2, 8, 24, 96, 4, 3, 70, 10),
    (1, 16, 3, 12, 10, 128, 8, 2, 90, 0), (1, 48, 2, 8, 8, 200, 4, 1, 64, 5), (3, 64, 2, 8, 8, 192, 8, 2, 80, 0),
    (3, 16, 3, 4, 8, 64, 4, 1, 33, 1), (0, 8, 2, 4, 6, 40, 4, 2, 50, 7),
]


@pytest.mark.parametrize("case", GS_CASES, ids=lambda c: "f%d_gs%d_K%d_S%d" % (c[0], c[1], c[5], c[7]))
def test_mla_group_scaled_weights(q, case):
    """Wkv_b with group-wise scales (one per row and gs columns), every format."""
    fmt, gs, H, Dn, Dv, K, R, S, T, st0 = case
    got, ref, bound = _run(q, fmt, H, Dn, Dv, K, R, S, T, st0, 0.3, seed=gs + K, gs=gs)
    assert_within(got.reshape(S, -1), ref.reshape(S, -1), bound.reshape(S, -1), TOL_F32, str(case))


def test_mla_full_size_int4_group_scaled(q):
    """64 heads, latent 512 + rope 64, 4096 positions, int4 Wkv_b with gs = 128."""
    H, Dn, Dv, K, R, T, S = 64, 128, 128, 512, 64, 4096, 1
    got, ref, bound = _run(q, 2, H, Dn, Dv, K, R, S, T, 0, (Dn + R) ** -0.5, seed=9, garbage=False, gs=128)
    assert_within(got.reshape(S, -1), ref.reshape(S, -1), bound.reshape(S, -1), TOL_F32, "full gs")


def test_bounded_wait_reports_timeout_and_context_survives(q):
    """A wait that runs out (an mbarrier nothing arrives on, 2 ms limit) is
    reported once by b200q_device_status; the next calls run normally."""
    import torch
    q.device_status()                                   # start from a clean record
    q.selftest_timeout(2000)
    with pytest.raises(q.B200QError) as ei:
        q.device_status()
    assert ei.value.status == q.ETIMEOUT
    assert q.device_status() == q.OK                    # cleared
    fmt, O, I = 2, 64, 256
    codes, sc = synth.quant_tensor(fmt, O, I, 0, 1, 5e-3, 2e-2)
    x = synth.activations(1, I, 0, 2)
    y_ref, bound = oracle.matmul(fmt, O, I, codes, sc, x)
    with q.tensor_upload(fmt, O, I, codes, sc) as t:
        y = torch.empty((1, O), dtype=torch.float32, device="cuda")
        q.matmul(t, to_dev(x), y, 1)
        torch.cuda.synchronize()
        assert_within(y.cpu().numpy(), y_ref, bound, TOL_F32, "after timeout")
    assert q.device_status() == q.OK
