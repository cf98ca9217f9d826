"""Pins of the CPU oracle against facts fixed outside it.

Each test checks the oracle against something other than itself: values
worked by hand from the pages' definitions (tests/golden/), examples whose
result depends on the summation order, exact integer sums, brute force over
tiny inputs, closed forms and library routines (numpy's binary16
conversions, Python's exact fsum).  A plausible slip in the oracle (a dropped
term, a wrong sign or index, another tree pairing, a transposed operand, a
residual added at the wrong place) fails at least one of them.
"""

import itertools
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from gradient_aggregation_gb300 import workload
from tests.conftest import read_golden


# ---- binary16 conversions ----------------------------------------------------

def test_half_to_float_all_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle.half_to_float(int(b)) for b in bits], dtype=np.float32)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin].view(np.uint32), ref[fin].view(np.uint32))
    assert np.array_equal(np.isinf(got), np.isinf(ref))
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_float_to_half_rne_matches_numpy():
    rng = np.random.default_rng(5)
    h = np.arange(0, 0x7c00, dtype=np.uint16).view(np.float16).astype(np.float32)
    # every finite fp16 value, its neighbours in fp32, and the midpoints
    mids = ((h[:-1].astype(np.float64) + h[1:]) / 2).astype(np.float32)
    cand = np.concatenate([
        h, np.nextafter(h, np.float32(np.inf)), np.nextafter(h, np.float32(0)),
        mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(np.inf)),
        np.float32([65504, 65519.99, 65520, 65536, 1e30, np.inf, 2.0 ** -25,
                    2.0 ** -26, 3 * 2.0 ** -26]),
        rng.standard_normal(20000).astype(np.float32) * np.float32(3000),
        (rng.standard_normal(20000) * 1e-5).astype(np.float32),
    ])
    cand = np.concatenate([cand, -cand])
    ref = cand.astype(np.float16).view(np.uint16)
    got = np.array([oracle.float_to_half(float(x)) for x in cand], dtype=np.uint16)
    assert np.array_equal(got, ref)


# ---- a1: layout and fusion -----------------------------------------------------

def test_alexnet_offsets_hand_worked():
    rows = read_golden("alexnet_offsets.txt")
    sizes = [int(r[1]) for r in rows[:-1]]
    expect = [int(r[2]) for r in rows[:-1]]
    assert tuple(sizes) == workload.get("alexnet").sizes
    off, n = oracle.layout(sizes)
    assert list(off) == expect
    assert n == int(rows[-1][1])


def test_fuse_pack_bitwise_round_trip():
    rng = np.random.default_rng(1)
    W, sizes = 3, [5, 1, 17, 8, 3]
    grads = [[rng.integers(0, 65536, n, dtype=np.uint16).view(np.float16)
              for n in sizes] for _ in range(W)]
    fused = oracle.fuse_pack(grads)
    assert fused.shape == (W, sum(sizes))
    # slice the fused rows back with numpy's own cumulative sum
    bounds = np.concatenate([[0], np.cumsum(sizes)])
    for w in range(W):
        for l, n in enumerate(sizes):
            seg = fused[w, bounds[l]:bounds[l + 1]]
            assert np.array_equal(seg.view(np.uint16), grads[w][l].view(np.uint16))


# ---- a2: tree order ---------------------------------------------------------------

def test_tree_order_discriminating_example():
    # 32768 + 2^-10 rounds back to 32768 in binary32 (ulp there is 2^-8).
    x = [32768.0, 2.0 ** -10, -32768.0, 2.0 ** -10]
    assert oracle.tree_sum(x) == 0.0          # ((x0+x1) + (x2+x3))
    # other orders give other answers, so the pin is discriminating
    seq = np.float32(0)
    for v in x:
        seq = np.float32(seq + np.float32(v))
    assert seq == 2.0 ** -10                   # sequential (parameter server)
    stride = np.float32(np.float32(x[0] + x[2]) + np.float32(x[1] + x[3]))
    assert stride == 2.0 ** -9                 # stride pairing


def test_tree_odd_counts_carry_last_element_up():
    t = 3 * 2.0 ** -11                          # 0.375 ulp of 2^15
    # W = 3: (x0 + x1) + x2 keeps 2^15; x0 + (x1 + x2) would give 2^15 + 2^-8
    assert oracle.tree_sum([32768.0, t, t]) == 32768.0
    # W = 5: ((x0+x1) + (x2+x3)) + x4 = 2^15 + 2^-8
    assert oracle.tree_sum([32768.0, t, t, t, t]) == 32768.0 + 2.0 ** -8
    # W = 6: ((x0+x1)+(x2+x3)) + (x4+x5)
    assert oracle.tree_sum([32768.0, t, t, t, t, t]) == 32768.0 + 2.0 ** -7


def _stack_order_sum(x):
    """Binary-counter form of the same tree: merge equal-height partial sums
    as leaves arrive, then fold the leftovers from the lowest height up."""
    stack = []  # (height, value)
    for v in x:
        h, val = 0, np.float32(v)
        while stack and stack[-1][0] == h:
            _, left = stack.pop()
            val = np.float32(left + val)
            h += 1
        stack.append((h, val))
    acc = stack.pop()[1]
    while stack:
        acc = np.float32(stack.pop()[1] + acc)
    return acc


@pytest.mark.parametrize("W", list(range(1, 20)) + [31, 32, 33, 63, 64, 65])
def test_tree_matches_binary_counter_form(W):
    rng = np.random.default_rng(W)
    for _ in range(200):
        # wide dynamic range so that grouping changes the rounding
        x = (rng.standard_normal(W) * np.exp(rng.uniform(-8, 8, W))).astype(np.float32)
        assert oracle.tree_sum(x) == _stack_order_sum(x)


def test_tree_reduce_exact_integer_sums_and_unscale():
    rng = np.random.default_rng(2)
    for W in (1, 2, 3, 5, 8, 16, 64):
        N = 37
        vals = rng.integers(-2048, 2049, size=(W, N))
        fused = vals.astype(np.float16)          # integers |v| <= 2048 are exact
        S = 256.0
        a = oracle.tree_reduce(fused, S)
        for i in range(N):
            exact = Fraction(int(vals[:, i].sum())) / (Fraction(S) * W)
            # the unscale is exact when S*W is a power of two
            if (W & (W - 1)) == 0:
                assert Fraction(float(a[i])) == exact
            else:
                assert abs(float(a[i]) - float(exact)) <= abs(float(exact)) * 2 ** -23


def _round_f32(x: Fraction) -> float:
    """The binary32 value nearest a positive rational in the normal range
    (ties to even), from the format's definition: 24 significant bits."""
    e = x.numerator.bit_length() - x.denominator.bit_length()
    if Fraction(2) ** e > x:
        e -= 1
    scale = Fraction(2) ** (e - 23)               # one unit in the last place
    m = x / scale                                 # in [2^23, 2^24)
    q, r = divmod(m.numerator, m.denominator)
    rem = Fraction(r, m.denominator)
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and q % 2 == 1):
        q += 1
    return float(q * scale)


def test_unscale_factor_is_the_nearest_binary32_to_one_over_s_w():
    """u = 1/(S*W) rounded once to binary32, also where S*W is not a power
    of two; S is the binary32 loss scale the calls take (1e-3 is first
    rounded to binary32)."""
    for S, W in [(1000.0, 3), (1024.0, 5), (512.0, 7), (65536.0, 6), (0.5, 3), (128.0, 96),
                 (3.0, 11), (1e-3, 13), (4096.0, 1), (256.0, 16)]:
        want = _round_f32(1 / (Fraction(float(np.float32(S))) * W))
        assert float(oracle.unscale_factor(S, W)) == want, (S, W)


def test_tree_reduce_worker_index_and_residual():
    # worker w contributes only element w: a transposed operand would fail
    W, N = 4, 4
    fused = np.zeros((W, N), dtype=np.float16)
    for w in range(W):
        fused[w, w] = 2.0 ** (w + 2)
    r = np.array([0.5, -0.25, 0.0, 1.0], dtype=np.float32)
    a = oracle.tree_reduce(fused, 1.0, r)
    expect = np.array([4 / 4 + 0.5, 8 / 4 - 0.25, 16 / 4, 32 / 4 + 1.0], dtype=np.float32)
    assert np.array_equal(a, expect)


def test_single_worker_is_plain_unscale():
    rng = np.random.default_rng(3)
    g = (rng.standard_normal(100) * 100).astype(np.float16)
    a = oracle.tree_reduce(g[None, :], 128.0)
    assert np.array_equal(a, g.astype(np.float32) / np.float32(128.0))


# ---- a2: other summation orders --------------------------------------------------

def test_sequential_order_discriminating_example():
    x = [32768.0, 2.0 ** -10, -32768.0, 2.0 ** -10]
    assert oracle.sequential_sum(x) == 2.0 ** -10   # (((x0+x1)+x2)+x3)
    t = 3 * 2.0 ** -11
    assert oracle.sequential_sum([t, t, 32768.0]) == 32768.0 + 2.0 ** -8
    assert oracle.sequential_sum([32768.0, t, t]) == 32768.0


def test_ring_segments_split_evenly():
    # N = 10, W = 4: boundaries floor(s*10/4) = 0, 2, 5, 7, 10
    assert [oracle.ring_segment(i, 10, 4) for i in range(10)] == [0, 0, 1, 1, 1, 2, 2, 3, 3, 3]
    assert [oracle.ring_segment(i, 3, 3) for i in range(3)] == [0, 1, 2]
    assert [oracle.ring_segment(i, 2, 5) for i in range(2)] == [2, 4]


def test_ring_order_hand_worked():
    # W = 3, N = 3: element i lies in segment i, so its sum starts at worker i.
    t = 3 * 2.0 ** -11                  # 0.375 ulp of 2^15
    big = 32768.0
    # element 0: ((x0 + x1) + x2) with x = [big, t, t]       -> big (t lost twice)
    # element 1: ((x1 + x2) + x0) with x = [big, t, t]       -> (2t = 0.75 ulp) + big = big + 2^-8
    # element 2: ((x2 + x0) + x1) with x = [t, t, big]       -> (big + t) + t = big
    col = [[big, t, t], [big, t, t], [t, t, big]]
    fused = np.array(col, dtype=np.float16).T.copy()        # fused[w, i]
    a = oracle.reduce_ordered(fused, 1.0, None, oracle.ORDER_RING)
    u = oracle.unscale_factor(1.0, 3)
    assert a[0] == np.float32(np.float32(big) * u)
    assert a[1] == np.float32(np.float32(big + 2.0 ** -8) * u)
    assert a[2] == np.float32(np.float32(big) * u)
    # the same columns in parameter-server order all start at worker 0
    s = oracle.reduce_ordered(fused, 1.0, None, oracle.ORDER_SEQUENTIAL)
    assert s[0] == np.float32(np.float32(big) * u)
    assert s[1] == np.float32(np.float32(big) * u)            # (big + t) + t
    assert s[2] == np.float32(np.float32(big + 2.0 ** -8) * u)  # (t + t) + big
    # and the tree order equals tree_reduce
    rng = np.random.default_rng(12)
    f = (rng.standard_normal((5, 50)) * 1000).astype(np.float16)
    assert np.array_equal(oracle.reduce_ordered(f, 8.0, None, 0), oracle.tree_reduce(f, 8.0))


def test_all_orders_agree_on_exact_integer_sums():
    rng = np.random.default_rng(13)
    vals = rng.integers(-2048, 2049, size=(7, 41))
    f = vals.astype(np.float16)
    outs = [oracle.reduce_ordered(f, 64.0, None, o) for o in (0, 1, 2)]
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


# ---- a3: norms ------------------------------------------------------------------

def test_norm_of_constant_chunk_is_closed_form():
    v = np.float32(0.3)
    a = np.full(256 * 3, v, dtype=np.float32)
    a[256:512] = -2.5
    n = oracle.chunk_norms(a, 256)
    assert n[0] == np.float32(16 * float(v))
    assert n[1] == np.float32(40.0)
    assert n[2] == np.float32(16 * float(v))


def test_norms_brute_force_with_partial_last_chunk():
    rng = np.random.default_rng(4)
    for N, cs in [(10, 4), (1, 1), (7, 7), (8, 3), (1000, 33)]:
        a = (rng.standard_normal(N) * np.exp(rng.uniform(-5, 5, N))).astype(np.float32)
        n = oracle.chunk_norms(a, cs)
        assert n.size == math.ceil(N / cs)
        for c in range(n.size):
            seg = [float(x) for x in a[c * cs:(c + 1) * cs]]
            exact = math.sqrt(math.fsum(x * x for x in seg))   # x*x exact in double
            assert abs(float(n[c]) - exact) <= exact * 2 ** -23


# ---- a4: selection ----------------------------------------------------------------

def _brute_force_kept(norms, k):
    """The unique k-subset in which every kept chunk beats every unkept one:
    larger norm, or equal norm and lower index."""
    C = len(norms)
    found = []
    for sub in itertools.combinations(range(C), k):
        s = set(sub)
        if all((norms[c] > norms[d]) or (norms[c] == norms[d] and c < d)
               for c in s for d in range(C) if d not in s):
            found.append(sub)
    assert len(found) == 1
    return list(found[0])


def test_select_brute_force_with_ties():
    rng = np.random.default_rng(6)
    for trial in range(300):
        C = int(rng.integers(1, 11))
        k = int(rng.integers(1, C + 1))
        pool = np.float32([0.0, 0.5, 1.0, 1.0, 2.0, 3.25])
        norms = rng.choice(pool, C) if trial % 2 else rng.random(C).astype(np.float32)
        norms = norms.astype(np.float32)
        idx, mask, _, thr = oracle.chunk_select(norms, k, want_packed=False)
        kept = _brute_force_kept([float(x) for x in norms], k)
        assert list(idx) == kept
        assert mask.sum() == k and all(mask[c] == 1 for c in kept)
        assert thr == min(norms[c] for c in kept)


def test_select_packed_is_kept_chunks_zero_padded():
    a = np.arange(1, 11, dtype=np.float32)       # N = 10, chunk 4 -> 3 chunks
    norms = oracle.chunk_norms(a, 4)             # last chunk [9, 10] is largest
    idx, mask, packed, thr = oracle.chunk_select(norms, 2, a, 4)
    assert list(idx) == [1, 2]
    assert list(mask) == [0, 1, 1]
    assert list(packed) == [5, 6, 7, 8, 9, 10, 0, 0]
    assert thr == norms[1]


def test_fp16_send_buffer_matches_numpy_rounding():
    rng = np.random.default_rng(11)
    packed = np.concatenate([
        (rng.standard_normal(5000) * np.exp(rng.uniform(-20, 12, 5000))).astype(np.float32),
        np.float32([0.0, -0.0, 65504.0, 70000.0, 1e-9, 2.0 ** -25])])
    for scale in (1.0, 512.0, 3.0):
        want = (packed * np.float32(scale)).astype(np.float16).view(np.uint16)
        assert np.array_equal(oracle.pack_fp16(packed, scale), want)
    # hand values: 1.5 * 2 = 3 exactly; 65504 * 2 overflows to +inf
    assert list(oracle.pack_fp16(np.float32([1.5, 65504.0, 0.0]), 2.0)) == [0x4200, 0x7c00, 0]


def test_keep_counts_hand_worked():
    for name, N, cs, C, p, k, last in read_golden("workload_counts.txt"):
        wl = workload.get(name)
        assert wl.N == int(N) and wl.chunk == int(cs) and wl.keep_percent == int(p)
        assert oracle.num_chunks(wl.N, wl.chunk) == int(C)
        assert oracle.keep_count(int(C), int(p), 100) == int(k)
        assert wl.N - (int(C) - 1) * wl.chunk == int(last)
    assert oracle.keep_count(3, 1, 1000) == 1       # never below one chunk


# ---- a5 and the whole step: hand-worked examples ----------------------------------

def _parse_hand(name):
    rows = read_golden(name)
    hdr, steps = {}, []
    for r in rows:
        if r[0] == "step":
            d, key, vals = {"step": int(r[1])}, None, []
            for tok in r[2:]:
                if tok in ("a", "kept", "r", "v", "w"):
                    if key:
                        d[key] = vals
                    key, vals = tok, []
                else:
                    vals.append(float(tok))
            d[key] = vals
            steps.append(d)
        else:
            hdr[r[0]] = [float(x) for x in r[1:]]
    return hdr, steps


def _run_hand(name, exact):
    hdr, steps = _parse_hand(name)
    W, cs = int(hdr["W"][0]), int(hdr["chunk"][0])
    g = [[np.float16(hdr["g0"])], [np.float16(hdr["g1"])]]
    g = [[np.asarray(hdr["g%d" % w], dtype=np.float16)] for w in range(W)]
    st = oracle.State(np.asarray(hdr["w0"], dtype=np.float32))
    k = int(hdr["k"][0])
    for d in steps:
        out = oracle.step(g, st, hdr["loss_scale"][0], cs, k, 2, hdr["lr"][0],
                          hdr["momentum"][0])
        assert out["k"] == k
        assert list(out["idx"]) == [int(x) for x in d["kept"]], d["step"]
        for key, arr in (("a", out["a"]), ("r", st.residual), ("v", st.velocity),
                         ("w", st.weights)):
            if key not in d:
                continue
            want = np.asarray(d[key], dtype=np.float64)
            if exact:
                assert np.array_equal(arr.astype(np.float64), want), (d["step"], key)
            else:
                assert np.allclose(arr, want, rtol=1e-6, atol=1e-7), (d["step"], key)


def test_hand_example_dyadic_exact():
    _run_hand("hand_2w2c_dyadic.txt", exact=True)


def test_hand_example_caffe_settings():
    _run_hand("hand_2w2c_caffe.txt", exact=False)


def test_partition_invariant_and_special_cases():
    rng = np.random.default_rng(7)
    N, cs = 1000, 64
    a = (rng.standard_normal(N)).astype(np.float32)
    C = oracle.num_chunks(N, cs)
    mask = (rng.random(C) < 0.3).astype(np.uint8)
    r = np.zeros(N, np.float32)
    v = (rng.standard_normal(N) * 0.1).astype(np.float32)
    w = rng.standard_normal(N).astype(np.float32)
    v0, w0 = v.copy(), w.copy()
    w16 = oracle.residual_sgd_update(a, mask, cs, 0.01, 0.0, r, v, w, want_w16=True)
    kept = np.repeat(mask, cs)[:N].astype(bool)
    g = np.where(kept, a, np.float32(0))
    # kept mass + residual mass = input, exactly one of them carries each value
    assert np.array_equal(np.where(kept, g, r), a)
    assert np.all((g == 0) | (r == 0))
    # momentum 0: v = lr*g, w = w - lr*g
    assert np.array_equal(v, np.float32(0.01) * g)
    assert np.array_equal(w, (w0 - np.float32(0.01) * g).astype(np.float32))
    assert np.array_equal(w16, w.astype(np.float16).view(np.uint16))
    # keeping everything leaves no residual
    r2 = np.ones(N, np.float32)
    oracle.residual_sgd_update(a, np.ones(C, np.uint8), cs, 0.01, 0.9, r2,
                               v0.copy(), w0.copy())
    assert not r2.any()


def test_update_accepts_residual_aliasing_a():
    rng = np.random.default_rng(8)
    N, cs = 100, 10
    a = rng.standard_normal(N).astype(np.float32)
    mask = np.array([1, 0] * 5, dtype=np.uint8)
    r1, v1, w1 = np.zeros(N, np.float32), np.zeros(N, np.float32), np.ones(N, np.float32)
    oracle.residual_sgd_update(a, mask, cs, 0.1, 0.9, r1, v1, w1)
    r2, v2, w2 = a.copy(), np.zeros(N, np.float32), np.ones(N, np.float32)
    oracle.residual_sgd_update(r2, mask, cs, 0.1, 0.9, r2, v2, w2)
    assert np.array_equal(r1, r2) and np.array_equal(v1, v2) and np.array_equal(w1, w2)


def test_keep_all_reduces_to_plain_tree_allreduce_sgd():
    rng = np.random.default_rng(9)
    W, sizes = 3, [50, 13]
    grads = [[(rng.standard_normal(n) * 100).astype(np.float16) for n in sizes]
             for _ in range(W)]
    st = oracle.State(np.ones(63, np.float32))
    out = oracle.step(grads, st, 64.0, 8, 100, 100, 0.1, 0.9)
    assert out["k"] == 8 and out["mask"].all()
    assert not st.residual.any()
    assert np.array_equal(st.weights, (np.float32(1) - np.float32(0.1) * out["a"]))


def test_step_is_deterministic():
    wl = workload.custom(W=5, sizes=[300, 77, 1000], chunk=64, keep_percent=20)
    grads = workload.all_grads(wl, 0)
    outs = []
    for _ in range(2):
        st = oracle.State(workload.initial_weights(wl))
        o = oracle.step(grads, st, wl.loss_scale, wl.chunk, 20, 100, wl.lr, wl.momentum)
        outs.append((o["a"].tobytes(), o["idx"].tobytes(), st.weights.tobytes()))
    assert outs[0] == outs[1]
