"""Pins the CPU oracle to what the pages and the mathematics fix.

Every check here comes from outside the oracle: values printed on the pages
(tests/golden/), library routines that implement the same special case (numpy's
stable sort, scipy's softmax, torch's bf16 / float8 casts), closed forms with
their error bounds, invariants the pages state, and brute force over every
routing of a tiny problem.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
from golden_io import payload_example, scan_example, worked_example

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def bf16_bits(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def bits_to_f32(b):
    return (np.asarray(b, np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------
def test_bf16_rne_matches_torch_cast():
    rng = np.random.default_rng(11)
    vals = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 4000),
        # exact ties: low 16 bits 0x8000 with even and odd upper halves
        (np.arange(0x3F80, 0x3F80 + 64, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
        (np.arange(0xBF80, 0xBF80 + 64, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
        np.array([0.0, -0.0, 3.3895313892515355e38, 1e-40, -1e-40], np.float32),
    ]).astype(np.float32)
    want = bf16_bits(vals)
    got = np.array([oracle.bf16_from_f32(float(v)) for v in vals], np.uint16)
    assert np.array_equal(got, want)
    for h in [0x0000, 0x8000, 0x3F80, 0xC2F7, 0x7F7F, 0x0001]:
        assert oracle.f32_from_bf16(h) == float(bits_to_f32([h])[0])


def test_e4m3_decode_matches_torch_for_every_code():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.e4m3_value(c)
        if (c & 0x7F) == 0x7F:
            assert math.isnan(got)
        else:
            assert got == ref[c], hex(c)
    # the format's fixed points: largest finite, smallest normal and subnormal
    assert oracle.e4m3_value(0x7E) == 448.0
    assert oracle.e4m3_value(0x08) == 2.0 ** -6
    assert oracle.e4m3_value(0x01) == 2.0 ** -9


def test_e4m3_encode_matches_torch_rne_below_saturation():
    rng = np.random.default_rng(12)
    reps = np.array([oracle.e4m3_value(c) for c in range(0x7F)], np.float64)
    mids = (reps[:-1] + reps[1:]) / 2  # exact ties
    vals = np.concatenate([
        rng.uniform(-447.0, 447.0, 3000), rng.standard_normal(3000) * 0.01,
        rng.standard_normal(1000) * 2.0 ** -8, reps, -reps, mids, -mids,
        np.nextafter(mids, 0), np.nextafter(mids, 1000)]).astype(np.float32)
    vals = vals[np.abs(vals) <= 448.0]
    want = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_from_f32(float(v)) for v in vals], np.uint8)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(vals[i]), hex(got[i]), hex(want[i])) for i in bad[:5]]


def test_e4m3_encode_saturates_and_keeps_sign():
    for v, code in [(448.0, 0x7E), (449.0, 0x7E), (1e6, 0x7E), (3e38, 0x7E), (-1e6, 0xFE),
                    (-0.0, 0x80), (0.0, 0x00), (-(2.0 ** -11), 0x80), (2.0 ** -11, 0x00),
                    (2.0 ** -10, 0x00),          # tie between 0 and 2^-9 -> even (0)
                    (3 * 2.0 ** -10, 0x02),      # tie between 1 and 2 (x 2^-9) -> even
                    (1.0625, 0x38), (1.1875, 0x3A)]:
        assert oracle.e4m3_from_f32(v) == code, (v, hex(oracle.e4m3_from_f32(v)))


# ---------------------------------------------------------------------------
# route
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("E,k,ties", [(256, 8, False), (64, 2, False), (8, 2, False),
                                       (256, 8, True), (33, 5, True), (1024, 32, False)])
def test_route_topk_matches_stable_sort_and_softmax(E, k, ties):
    from scipy.special import softmax
    rng = np.random.default_rng(E * 100 + k)
    T = 64
    if ties:
        z = rng.integers(-3, 4, (T, E)).astype(np.float32)  # many equal logits
    else:
        z = rng.standard_normal((T, E)).astype(np.float32)
    ids, w = oracle.route_topk(z, k)
    # numpy's stable sort of -z keeps the lower expert first among equal logits
    want_ids = np.argsort(-z, axis=1, kind="stable")[:, :k]
    assert np.array_equal(ids, want_ids)
    chosen = np.take_along_axis(z, want_ids, 1).astype(np.float64)
    want_w = softmax(chosen, axis=1).astype(np.float32)
    assert np.max(np.abs(w.view(np.int32) - want_w.view(np.int32))) <= 1
    # the renormalised full softmax is the same distribution
    full = softmax(z.astype(np.float64), axis=1)
    sel = np.take_along_axis(full, want_ids, 1)
    renorm = (sel / sel.sum(axis=1, keepdims=True)).astype(np.float32)
    assert np.max(np.abs(w.view(np.int32) - renorm.view(np.int32))) <= 2
    assert np.all(np.diff(w, axis=1) <= 0)


# ---------------------------------------------------------------------------
# layout
# ---------------------------------------------------------------------------
def test_layout_reproduces_worked_example():
    route, recv, na = worked_example()
    P, Tr, E, k = 4, 2, 8, 2
    ids = np.array([route[t] for t in range(8)], np.int32)
    assert ids.size == na == 16
    lay = oracle.layout(P, Tr, E, k, ids)
    x = np.zeros((8, 8), np.uint16)
    x[:, 0] = np.arange(8)  # row g carries g, so a receive row names its token
    rows, m = oracle.dispatch_bf16(P, Tr, E, k, x, np.ones((8, 2), np.float32), ids,
                                   lay["inv"], na)
    L = E // P
    for (r, e), tokens in recv.items():
        lo, hi = lay["expert_offset"][e], lay["expert_offset"][e + 1]
        got = [int(m["src_rank"][i]) * Tr + int(m["src_token"][i]) for i in range(lo, hi)]
        assert got == tokens, (r, e)
        assert list(rows[lo:hi, 0]) == tokens
        assert lay["rank_base"][r] <= lo and hi <= lay["rank_base"][r + 1]
        assert all(m["local_expert"][i] == e % L for i in range(lo, hi))
    assert list(lay["n_kept"]) == [2] * 8
    assert list(np.diff(lay["rank_base"])) == [4, 4, 4, 4]
    # per-source send counts of the worked routing (each column sums to 4)
    assert lay["C"].sum(axis=0).tolist() == [4, 4, 4, 4]
    assert lay["C"].sum(axis=1).tolist() == [4, 4, 4, 4]


def test_layout_reproduces_scan_example():
    counts, offsets = scan_example()
    # one source rank whose 4 tokens send 3, 1, 2, 2 assignments to ranks
    # 0..3 (E = 8, two experts per rank); the other ranks' slots are padding.
    P, Tr, E, k = 4, 4, 8, 2
    ids = -np.ones((P * Tr, k), np.int32)
    ids[0:4] = [[0, 1], [0, 2], [4, 6], [5, 7]]
    lay = oracle.layout(P, Tr, E, k, ids)
    assert lay["C"][0].tolist() == counts
    assert lay["send_offset"][0].tolist() == offsets
    assert lay["totals"].tolist() == [8, 0, P * Tr * k - 8]


def check_layout_invariants(P, Tr, E, k, ids, cap, lay):
    """The pages' invariants, checked row by row from the outputs."""
    L = E // P
    flat = ids.reshape(-1)
    Na = flat.size
    valid = [(a, int(flat[a])) for a in range(Na) if 0 <= flat[a] < E]
    # capacity: per expert, the first cap assignments in (s, t, j) order are kept
    kept = set()
    per_e = {}
    for a, e in valid:
        per_e.setdefault(e, []).append(a)
    for e, lst in per_e.items():
        kept.update(lst if cap == 0 else lst[:cap])
    inv = lay["inv"]
    nk = len(kept)
    # bijection: every kept assignment has exactly one row, rows are 0..nk-1
    assert sorted(int(inv[a]) for a in kept) == list(range(nk))
    assert all(inv[a] == -1 for a in range(Na) if a not in kept)
    row_to_a = {int(inv[a]): a for a in kept}
    # rows ordered by (expert, source, token, slot)
    keys = [(int(flat[row_to_a[r]]), row_to_a[r]) for r in range(nk)]
    assert keys == sorted(keys)
    # conservation: kept + dropped + masked = N_a
    masked = Na - len(valid)
    assert lay["totals"].tolist() == [nk, len(valid) - nk, masked]
    # ownership: rows of rank d hold experts owned by d
    for d in range(P):
        for r in range(lay["rank_base"][d], lay["rank_base"][d + 1]):
            assert int(flat[row_to_a[r]]) // L == d
    # expert segments and counts
    for e in range(E):
        lo, hi = lay["expert_offset"][e], lay["expert_offset"][e + 1]
        assert all(int(flat[row_to_a[r]]) == e for r in range(lo, hi))
        assert hi - lo == lay["n_kept"][e] and lay["n_raw"][e] == len(per_e.get(e, []))
    # count matrix, send and receive offsets, from the rows themselves
    C = np.zeros((P, P), int)
    for r in range(nk):
        a = row_to_a[r]
        C[(a // k) // Tr, int(flat[a]) // L] += 1
    assert np.array_equal(lay["C"], C)
    assert np.array_equal(lay["send_offset"], np.cumsum(C, axis=1) - C)
    for s in range(P):
        for e in range(E):
            lo = lay["expert_offset"][e]
            before = sum(1 for r in range(lo, lay["expert_offset"][e + 1])
                         if (row_to_a[r] // k) // Tr < s)
            assert lay["recv_offset"][s, e] == lo + before


def test_layout_brute_force_every_routing_tiny():
    """All 12^4 routings of P=2, T_r=2, E=4, k=2 (ordered distinct pairs), with
    no capacity and with capacity 1."""
    P, Tr, E, k = 2, 2, 4, 2
    pairs = [(a, b) for a in range(E) for b in range(E) if a != b]
    n = 0
    for combo in itertools.product(pairs, repeat=P * Tr):
        ids = np.array(combo, np.int32)
        for cap in (0, 1):
            lay = oracle.layout(P, Tr, E, k, ids, cap)
            if n % 97 == 0 or cap == 1 and n % 89 == 0:
                check_layout_invariants(P, Tr, E, k, ids, cap, lay)
            else:  # cheap subset of the invariants on every routing
                inv = lay["inv"]
                kept = inv[inv >= 0]
                assert sorted(kept.tolist()) == list(range(kept.size))
                assert lay["totals"][0] + lay["totals"][1] + lay["totals"][2] == ids.size
        n += 1
    assert n == 12 ** 4


@pytest.mark.parametrize("seed,cap,mask", [(1, 0, 0.0), (2, 3, 0.0), (3, 0, 0.2), (4, 2, 0.3)])
def test_layout_invariants_random(seed, cap, mask):
    rng = np.random.default_rng(seed)
    P, Tr, E, k = 3, 5, 6, 3
    ids = np.stack([rng.permutation(E)[:k] for _ in range(P * Tr)]).astype(np.int32)
    ids[rng.random(ids.shape) < mask] = -1
    lay = oracle.layout(P, Tr, E, k, ids, cap)
    check_layout_invariants(P, Tr, E, k, ids, cap, lay)


def test_layout_edge_cases():
    P, Tr, E, k = 4, 3, 8, 2
    # all tokens local: every token of rank s picks the two experts of rank s
    ids = np.array([[2 * (g // Tr), 2 * (g // Tr) + 1] for g in range(P * Tr)], np.int32)
    lay = oracle.layout(P, Tr, E, k, ids)
    assert np.array_equal(lay["C"], np.diag([Tr * k] * P))
    # all tokens to one remote rank (rank 3)
    ids = np.tile(np.array([[6, 7]], np.int32), (P * Tr, 1))
    lay = oracle.layout(P, Tr, E, k, ids)
    assert lay["C"][:, 3].tolist() == [Tr * k] * P and lay["C"][:, :3].sum() == 0
    assert lay["n_kept"][:6].sum() == 0  # empty experts
    # every slot masked
    lay = oracle.layout(P, Tr, E, k, -np.ones((P * Tr, k), np.int32))
    assert lay["totals"].tolist() == [0, 0, P * Tr * k] and (lay["inv"] == -1).all()
    # out-of-range ids are reported and treated as masked
    ids = np.array([[0, 1]] * (P * Tr), np.int32)
    ids[0, 1] = 99
    ids[1, 0] = -5
    lay = oracle.layout(P, Tr, E, k, ids)
    assert lay["bad_ids"] == 2 and lay["totals"][2] == 2


# ---------------------------------------------------------------------------
# dispatch
# ---------------------------------------------------------------------------
def test_dispatch_bf16_rows_are_the_source_rows():
    rng = np.random.default_rng(5)
    P, Tr, E, k, H = 2, 7, 4, 2, 16
    ids = np.stack([rng.permutation(E)[:k] for _ in range(P * Tr)]).astype(np.int32)
    w = rng.random((P * Tr, k)).astype(np.float32)
    x = bf16_bits(rng.standard_normal((P * Tr, H)))
    lay = oracle.layout(P, Tr, E, k, ids, 3)
    rows, m = oracle.dispatch_bf16(P, Tr, E, k, x, w, ids, lay["inv"], P * Tr * k)
    nk = lay["totals"][0]
    for r in range(nk):
        g = m["src_rank"][r] * Tr + m["src_token"][r]
        j = m["slot"][r]
        assert np.array_equal(rows[r], x[g])
        assert lay["inv"][g * k + j] == r
        assert m["local_expert"][r] == ids[g, j] % (E // P) and m["weight"][r] == w[g, j]


def test_dispatch_fp8_rows_scales_and_metadata():
    """The FP8 dispatch's placement, pinned row by row from outside the
    dispatch: every kept assignment a = (g, j) with row r = inv[a] holds the
    quantised token row (codes and scales of the separately pinned per-row
    quantiser) at payload row r and scale row r, and the metadata named by the
    pages' payload schema (local expert, source rank and token, slot, weight);
    rows at or beyond the kept count keep their fill. The ids are masked in
    places and a capacity drops rows, so some tokens have every slot dropped
    and some only a few."""
    rng = np.random.default_rng(15)
    P, Tr, E, k, H = 3, 11, 6, 3, 384  # three 128-channel blocks per row
    ids = np.stack([rng.permutation(E)[:k] for _ in range(P * Tr)]).astype(np.int32)
    ids[rng.random(ids.shape) < 0.2] = -1
    ids[4] = -1  # a token with every slot masked
    w = rng.random((P * Tr, k)).astype(np.float32)
    # each token row has its own scale per block, so a row or scale taken from
    # the wrong token or block cannot match
    mag = 10.0 ** rng.integers(-3, 3, (P * Tr, H // 128)).repeat(128, axis=1)
    x = bf16_bits(rng.standard_normal((P * Tr, H)) * mag)
    x[7, 128:256] = 0  # an all-zero block
    cap = 4
    lay = oracle.layout(P, Tr, E, k, ids, cap)
    inv = lay["inv"].reshape(P * Tr, k)
    rows = P * Tr * k
    q, sc, m = oracle.dispatch_fp8(P, Tr, E, k, x, w, ids, lay["inv"], rows)
    nk = int(lay["totals"][0])
    assert lay["totals"][1] > 0  # the capacity dropped something
    full_drop = [g for g in range(P * Tr)
                 if (ids[g] >= 0).any() and (inv[g] < 0).all()]
    partial = [g for g in range(P * Tr) if (inv[g] >= 0).any() and (inv[g] < 0).any()
               and (ids[g] >= 0).all()]
    assert full_drop and partial  # both kinds of token occur
    seen = np.zeros(rows, bool)
    for g in range(P * Tr):
        want_q, want_s = oracle.quantize_row_fp8(x[g])
        for j in range(k):
            r = int(inv[g, j])
            if r < 0:
                continue
            assert not seen[r]
            seen[r] = True
            assert np.array_equal(q[r], want_q), (g, j)
            assert np.array_equal(sc[r].view(np.uint32), want_s.view(np.uint32)), (g, j)
            assert m["local_expert"][r] == ids[g, j] % (E // P)
            assert m["src_rank"][r] == g // Tr and m["src_token"][r] == g % Tr
            assert m["slot"][r] == j and m["weight"][r] == w[g, j]
    assert seen[:nk].all() and not seen[nk:].any()
    # untouched fill past the kept rows
    assert not q[nk:].any() and not sc[nk:].any()
    for name in ("local_expert", "src_rank", "src_token", "slot"):
        assert (m[name][nk:] == -7).all()
    assert np.isnan(m["weight"][nk:]).all()


def test_token_range_threads_give_the_same_results():
    """The oracle's threads option only splits tokens across threads; every
    output must equal the single-threaded call's."""
    rng = np.random.default_rng(16)
    P, Tr, E, k, H = 3, 13, 12, 4, 256
    z = rng.standard_normal((P * Tr, E)).astype(np.float32)
    ids1, w1 = oracle.route_topk(z, k)
    ids4, w4 = oracle.route_topk(z, k, threads=4)
    assert np.array_equal(ids1, ids4) and np.array_equal(w1.view(np.int32), w4.view(np.int32))
    x = bf16_bits(rng.standard_normal((P * Tr, H)))
    lay = oracle.layout(P, Tr, E, k, ids1, 9)
    rows = P * Tr * k
    a = oracle.dispatch_fp8(P, Tr, E, k, x, w1, ids1, lay["inv"], rows)
    b = oracle.dispatch_fp8(P, Tr, E, k, x, w1, ids1, lay["inv"], rows, threads=5)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1].view(np.int32), b[1].view(np.int32))
    for n in a[2]:
        assert np.array_equal(a[2][n].view(np.int32), b[2][n].view(np.int32)), n
    c = oracle.dispatch_bf16(P, Tr, E, k, x, w1, ids1, lay["inv"], rows)
    d = oracle.dispatch_bf16(P, Tr, E, k, x, w1, ids1, lay["inv"], rows, threads=3)
    assert np.array_equal(c[0], d[0])
    for n in c[1]:
        assert np.array_equal(c[1][n].view(np.int32), d[1][n].view(np.int32)), n
    y1 = oracle.expert_dequant_fp8(a[0], a[1])
    y3 = oracle.expert_dequant_fp8(a[0], a[1], threads=3)
    assert np.array_equal(y1, y3)
    o1 = oracle.combine(lay["inv"], w1, y1, P * Tr, k)
    o6 = oracle.combine(lay["inv"], w1, y1, P * Tr, k, threads=6)
    assert np.array_equal(o1, o6)


def test_quantize_fp8_error_bound_and_closed_checks():
    rng = np.random.default_rng(6)
    H = 1024
    xs = rng.standard_normal(H).astype(np.float32) * 10.0 ** rng.integers(-3, 3, H // 128).repeat(128)
    xs[256:384] = 0.0  # an all-zero block
    xb = bf16_bits(xs)
    q, sc = oracle.quantize_row_fp8(xb)
    xf = bits_to_f32(xb).astype(np.float64)
    qv = np.array([oracle.e4m3_value(c) for c in q])
    assert sc[2] == 0.0 and not q[256:384].any()
    for b in range(H // 128):
        blk = slice(b * 128, (b + 1) * 128)
        amax = np.max(np.abs(xf[blk]))
        if amax == 0:
            continue
        s = float(np.float32(np.float32(amax) / np.float32(448.0)))
        assert sc[b] == s
        assert np.max(np.abs(qv[blk])) <= 448.0
        i = int(np.argmax(np.abs(xf[blk])))
        assert q[b * 128 + i] & 0x7F == 0x7E  # the amax element lands on +-448
        v = xf[blk] / s
        # half an e4m3 ulp at |v|: 2^(e-3)/2 for normals, 2^-10 for subnormals
        e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -6)))
        half_ulp = 2.0 ** (e - 4)
        err = np.abs(v - qv[blk])
        assert np.all(err <= half_ulp * (1 + 1e-6) + 1e-12), b
    # codes equal torch's RNE cast of the fp32 quotient (no saturation needed)
    for b in range(H // 128):
        if sc[b] == 0:
            continue
        quo = (bits_to_f32(xb[b * 128:(b + 1) * 128]) / np.float32(sc[b])).astype(np.float32)
        quo = np.clip(quo, -448, 448)
        want = torch.from_numpy(quo).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(q[b * 128:(b + 1) * 128], want)


# ---------------------------------------------------------------------------
# expert stand-ins and combine
# ---------------------------------------------------------------------------
def test_expert_standins_match_torch_arithmetic():
    rng = np.random.default_rng(7)
    E, H = 4, 256
    eoff = np.array([0, 3, 3, 7, 9], np.int32)
    c = (rng.random(E, dtype=np.float32) + np.float32(0.5)).astype(np.float32)
    x = bf16_bits(rng.standard_normal((9, H)))
    y = oracle.expert_scale_bf16(E, eoff, c, x)
    e_of_row = np.repeat(np.arange(E), np.diff(eoff))
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float()
    want = (xt * torch.from_numpy(c[e_of_row])[:, None]).to(torch.bfloat16)
    assert np.array_equal(y, want.view(torch.int16).numpy().view(np.uint16))
    q = rng.integers(0, 256, (5, H)).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x11  # no NaN codes
    s = rng.random((5, H // 128)).astype(np.float32)
    y = oracle.expert_dequant_fp8(q, s)
    qf = torch.from_numpy(q).view(torch.float8_e4m3fn).float()
    want = (qf * torch.from_numpy(np.repeat(s, 128, axis=1))).to(torch.bfloat16)
    assert np.array_equal(y, want.view(torch.int16).numpy().view(np.uint16))


def test_combine_identity_round_trip_closed_form():
    """Identity expert: out = bf16(sum_j w_j * x) within one bf16 ulp of the
    exact value; the worked example's 0.6/0.4 weights give back x."""
    route, _, _ = worked_example()
    P, Tr, E, k, H = 4, 2, 8, 2, 128
    ids = np.array([route[t] for t in range(8)], np.int32)
    rng = np.random.default_rng(8)
    x = bf16_bits(rng.standard_normal((8, H)))
    w = np.tile(np.array([0.6, 0.4], np.float32), (8, 1))
    lay = oracle.layout(P, Tr, E, k, ids)
    rows, _ = oracle.dispatch_bf16(P, Tr, E, k, x, w, ids, lay["inv"], 16)
    out = oracle.combine(lay["inv"], w, rows, 8, k)
    xf = bits_to_f32(x).astype(np.float64)
    of = bits_to_f32(out).astype(np.float64)
    ulp = 2.0 ** (np.floor(np.log2(np.abs(xf))) - 7)
    assert np.all(np.abs(of - xf) <= ulp)
    # general weights, k = 3, some slots masked
    rng = np.random.default_rng(9)
    P, Tr, E, k, H = 2, 9, 6, 3, 64
    ids = np.stack([rng.permutation(E)[:k] for _ in range(P * Tr)]).astype(np.int32)
    ids[rng.random(ids.shape) < 0.25] = -1
    w = rng.random((P * Tr, k)).astype(np.float32)
    x = bf16_bits(rng.standard_normal((P * Tr, H)))
    lay = oracle.layout(P, Tr, E, k, ids)
    rows, _ = oracle.dispatch_bf16(P, Tr, E, k, x, w, ids, lay["inv"], P * Tr * k)
    out = oracle.combine(lay["inv"], w, rows, P * Tr, k)
    wsum = np.where(ids >= 0, w, 0).astype(np.float64).sum(axis=1)
    exact = bits_to_f32(x).astype(np.float64) * wsum[:, None]
    of = bits_to_f32(out).astype(np.float64)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(exact), 1e-30))) - 7)
    assert np.all(np.abs(of - exact) <= ulp)
    assert np.all(out[wsum == 0] == 0)


def test_combine_uses_fused_multiply_add_in_slot_order():
    """A case where a fused and an unfused multiply-add differ. Slot 0 gives
    acc = -(1 + 2^-7) exactly; slot 1's exact product (1 + 2^-23)(1 + 2^-7) =
    1 + 2^-7 + 2^-23 + 2^-30 needs 31 bits, so only a single rounding of
    w1*y1 + acc keeps the 2^-30 term: the result is 2^-23 + 2^-30, whose bf16
    is 2^-23 * (1 + 2^-7); an unfused product would give exactly 2^-23."""
    y = bf16_bits(np.array([[1.0 + 2 ** -7], [1.0 + 2 ** -7]], np.float32))
    w = np.array([[-1.0, 1.0 + 2 ** -23]], np.float32)
    out = oracle.combine(np.array([0, 1], np.int32), w, y, 1, 2)
    assert out[0, 0] == bf16_bits(np.array([2.0 ** -23 * (1 + 2 ** -7)], np.float32))[0]
    # reversing the slots changes the operation order and the result
    out = oracle.combine(np.array([1, 0], np.int32), w[:, ::-1].copy(), y, 1, 2)
    assert out[0, 0] == bf16_bits(np.array([2.0 ** -23], np.float32))[0]


def test_payload_arithmetic_88mb():
    from combine_top_histogram_gb300.accounting import wire_payload_bytes
    d = payload_example()
    b = wire_payload_bytes(d["tokens"], d["top_k"], d["hidden"], d["dispatch_bytes"],
                           d["combine_bytes"])
    assert b == 2048 * 2 * 7168 * 3
    assert round(b / 1e6) == d["approx_mb"]
