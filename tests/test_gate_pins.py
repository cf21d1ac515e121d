"""CPU pins of the parity gates (oracle/gates.py): every GPU verdict passes through them.

Each gate is checked against something other than itself:
  * ulp_bf16 against the distance to the next bf16 value, decoded by torch from the bit
    pattern one above (every positive finite bf16, powers of two and subnormals included),
    and against binary64 values on both sides of each power of two;
  * check_bf16, check_f32_rel and check_dw at their boundaries (a value exactly at the
    tolerance passes, one just beyond it fails, in both directions and with NaN/inf);
  * dx_fp32_bound against a binary32 evaluation of dX in the order the library documents
    for its kernels (sequential per-lane FMA chains over even/odd element pairs, the two
    chains added, a 32-lane shuffle tree, each warp's part scaled by rstd^2/H, the parts
    added in warp order, then RN(rstd * fma(x, -c', RN(dy*w)))): the bound covers every
    element, including rows built for near-total cancellation; the same rows break the
    bound when its c' term is dropped (so they exercise it), and the worst error reaches a
    stated fraction of the bound (so it is not vacuous).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import gates

U = 2.0 ** -24


# ------------------------------------------------------------------------ ulp_bf16
def _bf16_values(bits):
    t = torch.from_numpy(np.asarray(bits, dtype=np.uint16).view(np.int16).copy())
    return t.view(torch.bfloat16).double().numpy()


def test_ulp_bf16_is_the_distance_to_the_next_bf16():
    bits = np.arange(0x0000, 0x7F7F, dtype=np.uint32)  # every positive finite bf16 but the max
    v = _bf16_values(bits)
    nxt = _bf16_values(bits + 1)
    spacing = nxt - v
    np.testing.assert_array_equal(gates.ulp_bf16(v), spacing)
    np.testing.assert_array_equal(gates.ulp_bf16(-v), spacing)
    assert gates.ulp_bf16(np.array([0.0]))[0] == 2.0 ** -133  # the subnormal quantum
    assert gates.ulp_bf16(np.array([2.0 ** -130]))[0] == 2.0 ** -133
    assert gates.ulp_bf16(np.array([2.0 ** -126]))[0] == 2.0 ** -133
    assert gates.ulp_bf16(np.array([1.0]))[0] == 2.0 ** -7


@pytest.mark.parametrize("k", [-126, -60, -1, 0, 1, 9, 10, 60, 127])
def test_ulp_bf16_on_both_sides_of_a_power_of_two(k):
    p = 2.0 ** k
    below = np.nextafter(p, 0.0)  # the largest binary64 value in the binade below
    assert gates.ulp_bf16(np.array([p]))[0] == 2.0 ** (k - 7)
    assert gates.ulp_bf16(np.array([below]))[0] == 2.0 ** (max(k - 1, -126) - 7)
    assert gates.ulp_bf16(np.array([np.nextafter(p, np.inf)]))[0] == 2.0 ** (k - 7)


def test_bf16_to_f64_decodes_every_pattern_like_torch():
    bits = np.arange(0, 1 << 16, dtype=np.uint32)
    ours = gates.bf16_to_f64(bits.astype(np.uint16))
    ref = _bf16_values(bits)
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[fin], ref[fin])


# ------------------------------------------------------------------------ check_bf16
def _bits(values):
    return torch.tensor(values, dtype=torch.float64).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def test_check_bf16_one_ulp_boundary():
    d = _bits([1.5, -1.5, 3.0])  # exact bf16 values
    ulp = np.array([2.0 ** -7, 2.0 ** -7, 2.0 ** -6])
    at = np.array([1.5, -1.5, 3.0]) - np.sign([1.5, -1.5, 3.0]) * ulp  # refs exactly 1 ulp away
    r = gates.check_bf16(d, at)
    assert r["n_fail"] == 0 and r["max_err_in_ulp"] == 1.0 and r["n_widened"] == 0
    beyond = at - np.sign(at) * 2.0 ** -30  # one ulp plus a sliver: outside
    r = gates.check_bf16(d, beyond)
    assert r["n_fail"] == 3 and r["first_fail"] == (0,)
    inside = at + np.sign(at) * 2.0 ** -30
    assert gates.check_bf16(d, inside)["n_fail"] == 0


def test_check_bf16_widening_is_counted_and_bounded():
    d = _bits([1.5, 1.5])
    ref = np.array([1.5 - 2.0 ** -7 - 2.0 ** -30, 1.5])
    r = gates.check_bf16(d, ref, extra=np.array([2.0 ** -29, 0.0]))
    assert r["n_fail"] == 0 and r["n_widened"] == 1 and r["frac_widened"] == 0.5
    r = gates.check_bf16(d, ref, extra=np.array([2.0 ** -31, 0.0]))
    assert r["n_fail"] == 1 and r["n_widened"] == 0
    # 2-D: the widened element's error on its row's scale (row rms ~1.5: ulp 2^-7)
    r = gates.check_bf16(d.reshape(1, 2), ref.reshape(1, 2), extra=np.array([[2.0 ** -29, 0.0]]))
    assert r["n_widened"] == 1
    assert r["max_widened_err_row_ulp"] == pytest.approx(1.0 + 2.0 ** -23)


def test_check_bf16_rejects_nan_and_inf():
    d = np.array([0x7FC0, 0x7F80, 0xFF80], dtype=np.uint16)  # NaN, +inf, -inf
    r = gates.check_bf16(d, np.array([1.0, 3e38, -3e38]), extra=np.full(3, 1e300))
    assert r["n_fail"] == 3


# ------------------------------------------------------------------------ check_f32_rel
def test_check_f32_rel_boundary():
    ref = np.array([1.0, -2.0, 1e-30])
    assert gates.check_f32_rel(ref * (1 + 0.999e-5), ref)["n_fail"] == 0
    assert gates.check_f32_rel(ref * (1 - 0.999e-5), ref)["n_fail"] == 0
    r = gates.check_f32_rel(ref * (1 + 1.001e-5), ref)
    assert r["n_fail"] == 3 and r["worst_ratio"] == pytest.approx(1.001, rel=1e-6)
    assert gates.check_f32_rel(np.array([np.nan]), np.array([1.0]))["n_fail"] == 1
    assert gates.check_f32_rel(np.array([0.0]), np.array([0.0]))["n_fail"] == 0


def test_check_f32_rel_row_rms_term():
    ref = np.array([[3.0, 4.0, 0.0, 0.0]])  # rms = 2.5
    d = ref.copy()
    d[0, 2] = 0.999e-5 * 2.5
    assert gates.check_f32_rel(d, ref, row_rms_term=True)["n_fail"] == 0
    assert gates.check_f32_rel(d, ref, row_rms_term=False)["n_fail"] == 1
    d[0, 2] = 1.001e-5 * 2.5
    assert gates.check_f32_rel(d, ref, row_rms_term=True)["n_fail"] == 1
    # the row term is per row: a second row with a tiny rms does not borrow the first's
    ref2 = np.vstack([ref, [[1e-3, 0.0, 0.0, 0.0]]])
    d2 = ref2.copy()
    d2[1, 1] = 1e-5 * 2.5 * 0.5
    assert gates.check_f32_rel(d2, ref2, row_rms_term=True)["n_fail"] == 1


# ------------------------------------------------------------------------ check_dw
def test_check_dw_budget_boundary():
    ref = np.array([0.0, 100.0, -100.0])
    tol = 1e-4 + 1e-4 * np.abs(ref)
    assert gates.check_dw(ref + 0.999 * tol, ref)["n_fail"] == 0
    assert gates.check_dw(ref - 0.999 * tol, ref)["n_fail"] == 0
    r = gates.check_dw(ref - 1.001 * tol, ref)
    assert r["n_fail"] == 3 and r["worst"] == pytest.approx(1.001, rel=1e-6)
    assert gates.check_dw(np.array([np.inf]), np.array([0.0]))["n_fail"] == 1
    assert gates.check_dw(np.array([np.nan]), np.array([0.0]))["n_fail"] == 1
    r = gates.check_dw(np.array([3.0, 4.0]) * 1.5, np.array([3.0, 4.0]))
    assert r["rel_l2"] == pytest.approx(0.5)


# --------------------------------------------------------------- dx_fp32_bound
def _f32(a):
    return np.asarray(a, dtype=np.float64).astype(np.float32)


def _fma32(a, b, c):
    # binary64 product (exact: at most 48 significant bits) plus c, rounded to binary64 then
    # binary32; the double rounding adds at most 2^-53 relative, inside gamma's slack
    return (np.asarray(a, np.float64) * np.asarray(b, np.float64) + np.asarray(c, np.float64)) \
        .astype(np.float32)


def _warp_tree(lane_vals):
    """Lane 0's value after the row-sum shuffles: lanes paired (l, l^1), then butterflies
    over lane distances 16, 8, 4, 2 (rows x 32 lanes in, rows out)."""
    s = lane_vals[:, 0::2] + lane_vals[:, 1::2]  # lane 2k: its own value plus lane 2k+1's
    idx = np.arange(16)
    for o in (8, 4, 2, 1):  # lane distances 16, 8, 4, 2 in the paired index
        s = s + s[:, idx ^ o]
    return s[:, 0]


def _scale(rs, H):
    return _f32(rs * _f32(rs * _f32(1.0 / H))).astype(np.float32)


def _dx_kernel_order(dy, x, w, rs, nw, nch, vec, small=False):
    """binary32 dX in the documented order.  Strip kernel: lane t of nw*32 holds the
    16-byte vectors c*nw*32 + t (c < nch).  Small-T kernel: 256 threads, thread t holds
    vectors t, t + 256, ...  (small=True; nw and nch are then derived)."""
    R, H = x.shape
    nvec = H // vec
    npair = vec // 2
    p = _f32(dy * x)
    w32 = _f32(w)
    if small:
        nw, threads = 8, 256
        per = -(-nvec // threads)
        vec_of = [[t + k * threads for k in range(per)] for t in range(threads)]
    else:
        threads = nw * 32
        vec_of = [[c * threads + t for c in range(nch)] for t in range(threads)]
    lane = np.zeros((R, threads), np.float32)
    for t in range(threads):
        lo = np.zeros(R, np.float32)
        hi = np.zeros(R, np.float32)
        for v in vec_of[t]:
            if v >= nvec:
                continue
            for i in range(npair):
                j = v * vec + 2 * i
                lo = _fma32(w32[j], p[:, j], lo)
                hi = _fma32(w32[j + 1], p[:, j + 1], hi)
        lane[:, t] = lo + hi
    m = _scale(rs, H)
    c = None
    for k in range(nw):
        post = (_warp_tree(lane[:, 32 * k:32 * k + 32]) * m).astype(np.float32)
        c = post if c is None else (c + post).astype(np.float32)
    g = _f32(dy * w[None, :])
    f = _fma32(x, -c[:, None].astype(np.float64), g)
    return (np.asarray(rs, np.float32)[:, None] * f).astype(np.float32), c


def _rows(H, n_rand, n_cancel, seed, x_bf16=True, w_bf16=True):
    rng = np.random.default_rng(seed)
    rnd = (lambda a: oracle.bf16_round(a).reshape(np.shape(a))) if x_bf16 else _f32
    dec = oracle.bf16_bits_to_f64 if x_bf16 else (lambda a: np.asarray(a, np.float64))
    w = 1.0 + 0.1 * rng.standard_normal(H)
    w = dec(oracle.bf16_round(w)) if w_bf16 else _f32(w).astype(np.float64)
    x = dec(rnd(rng.standard_normal((n_rand + n_cancel, H))))
    dy = rng.standard_normal((n_rand + n_cancel, H))
    ms = np.mean(x * x, axis=1)
    rs = _f32(1.0 / np.sqrt(ms + 1e-6)).astype(np.float64)
    # cancellation rows: dy proportional to xhat / w, so g - xhat*c nearly vanishes
    lam = rng.uniform(0.5, 4.0, size=n_cancel)
    dy[n_rand:] = lam[:, None] * x[n_rand:] * rs[n_rand:, None] / w[None, :] * \
        (1.0 + 1e-3 * rng.standard_normal((n_cancel, H)))
    dy = dec(rnd(dy))
    return dy, x, w, rs


# (H, consumer warps, vectors per lane) as the planner picks them for the strip kernel,
# and the small-T kernel's fixed 256-thread row task
GEOMETRIES = [(256, 1, 1, False), (1536, 3, 2, False), (2048, 4, 2, False),
              (2560, 5, 2, False), (3584, 7, 2, False), (4096, 8, 2, False),
              (6144, 8, 3, False), (4096, 8, 2, True)]


@pytest.mark.parametrize("H,nw,nch,small", GEOMETRIES)
@pytest.mark.parametrize("xbf", [True, False])
def test_dx_fp32_bound_covers_the_kernel_order(H, nw, nch, small, xbf):
    vec = 8 if xbf else 4
    if not xbf:
        nch = max(1, -(-(H // vec) // (nw * 32)))
    dy, x, w, rs = _rows(H, 24, 24, seed=H + nw + int(xbf), x_bf16=xbf, w_bf16=xbf)
    dx32, _ = _dx_kernel_order(dy, x, w, rs, nw, nch, vec, small=small)
    # exact dX (binary64 oracle, at the same saved rstd)
    enc = (lambda a: oracle.bf16_round(a).reshape(np.shape(a))) if xbf else _f32
    wenc = oracle.bf16_round(w) if xbf else _f32(w)
    dx_ref, _ = oracle.rmsnorm_bwd(enc(dy), enc(x), wenc, rs, want_dw=False)
    if small:
        chain = -(-(H // vec) // 256) * (vec // 2)
        depth = gates.row_dot_depth(chain, 8)
    else:
        depth = gates.row_dot_depth(nch * (vec // 2), nw)
    B = gates.dx_fp32_bound(dy, x, w, rs, dx_ref, depth)
    err = np.abs(dx32.astype(np.float64) - dx_ref)
    assert np.all(err <= B), float(np.max(err / B))
    # the bound is not vacuous: the worst error it must cover reaches a quarter of it over
    # all rows (measured 0.49-0.77), and 1/32 of it on the cancellation rows, where its c'
    # term dominates (measured 0.06-0.17)
    assert np.max(err / B) > 0.25
    assert np.max((err / B)[24:]) > 1.0 / 32.0
    # the cancellation rows need the c' term: without it the bound fails there
    r = rs[:, None]
    g = dy * w[None, :]
    no_c_term = gates.gamma(2) * np.abs(dx_ref) + (1 + gates.gamma(2)) * r * U * np.abs(g)
    assert np.any(err > no_c_term)


def test_row_dot_depth_counts_the_documented_tree():
    # 8 warps; each lane chains 2 bf16 vectors of 4 element pairs
    assert gates.row_dot_depth(2 * 4, 8) == 1 + 8 + 1 + 5 + 1 + 3 + 7
    assert gates.row_dot_depth(1, 1) == 1 + 1 + 1 + 5 + 1 + 3 + 0
    assert gates.gamma(1) == pytest.approx(U / (1 - U))
