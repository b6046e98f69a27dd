"""Pins of the K/V short-convolution + paged-write oracle (``oracle/kv_conv.py``) against
things other than itself: identity, exact shifts, a hand-worked example, numpy's own
convolution on integer data, chunking invariance, and mutants that must fail."""
import numpy as np
import pytest

import oracle.kv_conv as kc


def to_bits(x):
    return kc.f64_to_bf16_bits(np.asarray(x, np.float64))


def make_case(rng, *, B=3, Hkv=2, D=8, P=4, ks=4, n=(5, 1, 3), L=(5, 9, 12), integer=False):
    T = sum(n)
    cu = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    pages_per = [-(-l // P) for l in L]
    num_pages = sum(pages_per) + 2
    perm = rng.permutation(num_pages)
    bt = np.full((B, max(pages_per)), num_pages + 7, np.int32)
    c = 0
    for b, npg in enumerate(pages_per):
        bt[b, :npg] = perm[c:c + npg]
        c += npg
    draw = (lambda *s: rng.integers(-3, 4, s).astype(np.float64)) if integer else (lambda *s: rng.standard_normal(s))
    k_new, v_new = to_bits(draw(T, Hkv, D)), to_bits(draw(T, Hkv, D))
    st_k, st_v = to_bits(draw(B, ks - 1, Hkv, D)), to_bits(draw(B, ks - 1, Hkv, D))
    w_k, w_v = draw(Hkv, D, ks), draw(Hkv, D, ks)
    cache_k = to_bits(rng.standard_normal((num_pages, Hkv, P, D)))
    cache_v = to_bits(rng.standard_normal((num_pages, Hkv, P, D)))
    return dict(k_new_bits=k_new, v_new_bits=v_new, cu_q=cu, seq_lens=np.array(L, np.int32), block_table=bt,
                page_size=P, w_k=w_k, w_v=w_v, ks=ks, state_k_bits=st_k, state_v_bits=st_v,
                k_cache_bits=cache_k, v_cache_bits=cache_v)


def written_slots(case):
    P = case["page_size"]
    slots = set()
    for b in range(len(case["seq_lens"])):
        n = case["cu_q"][b + 1] - case["cu_q"][b]
        L = case["seq_lens"][b]
        for i in range(n):
            p = L - n + i
            slots.add((int(case["block_table"][b][p // P]), p % P))
    return slots


def test_identity_kernel_writes_the_raw_rows_and_nothing_else():
    rng = np.random.default_rng(0)
    case = make_case(rng, ks=1)
    case["w_k"] = np.ones_like(case["w_k"])
    case["w_v"] = np.ones_like(case["w_v"])
    kc_, vc_, sk, sv = kc.kv_conv_write(**case)
    P = case["page_size"]
    for b in range(3):
        t0, t1 = case["cu_q"][b], case["cu_q"][b + 1]
        L = case["seq_lens"][b]
        for i, t in enumerate(range(t0, t1)):
            p = L - (t1 - t0) + i
            pg = case["block_table"][b][p // P]
            assert np.array_equal(kc_[pg, :, p % P], case["k_new_bits"][t])
            assert np.array_equal(vc_[pg, :, p % P], case["v_new_bits"][t])
    ws = written_slots(case)
    for pg in range(kc_.shape[0]):
        for s in range(P):
            if (pg, s) not in ws:
                assert np.array_equal(kc_[pg, :, s], case["k_cache_bits"][pg, :, s])
    assert sk.shape[1] == 0 and sv.shape[1] == 0


@pytest.mark.parametrize("j", [0, 1, 3])
def test_one_hot_kernel_is_an_exact_shift_through_the_state(j):
    check_one_hot_shift(kc, j)


def check_one_hot_shift(kc, j):
    rng = np.random.default_rng(1 + j)
    ks = 4
    case = make_case(rng, ks=ks)
    w = np.zeros_like(case["w_k"])
    w[:, :, j] = 1.0
    case["w_k"] = case["w_v"] = w
    kc_, _, _, _ = kc.kv_conv_write(**case)
    P = case["page_size"]
    for b in range(3):
        t0, t1 = case["cu_q"][b], case["cu_q"][b + 1]
        n, L = t1 - t0, case["seq_lens"][b]
        hist = np.concatenate([case["state_k_bits"][b], case["k_new_bits"][t0:t1]], axis=0)
        for i in range(n):
            p = L - n + i
            src = hist[i + j]  # position p - (ks - 1) + j
            pg = case["block_table"][b][p // P]
            assert np.array_equal(kc_[pg, :, p % P], src)


def test_hand_worked_example():
    check_hand_worked(kc)


def check_hand_worked(kc):
    # one sequence, one channel, ks 3, w = (1, 2, 4), state (10, 20), new inputs (1, 2, 3):
    # y(p0) = 1*10 + 2*20 + 4*1 = 54, y(p1) = 1*20 + 2*1 + 4*2 = 30, y(p2) = 1*1 + 2*2 + 4*3 = 17
    case = dict(k_new_bits=to_bits(np.array([1, 2, 3.0]).reshape(3, 1, 1)),
                v_new_bits=to_bits(np.zeros((3, 1, 1))), cu_q=np.array([0, 3], np.int32),
                seq_lens=np.array([7], np.int32), block_table=np.array([[2, 0]], np.int32), page_size=4,
                w_k=np.array([1, 2, 4.0]).reshape(1, 1, 3), w_v=np.zeros((1, 1, 3)), ks=3,
                state_k_bits=to_bits(np.array([10, 20.0]).reshape(1, 2, 1, 1)),
                state_v_bits=to_bits(np.zeros((1, 2, 1, 1))),
                k_cache_bits=np.zeros((3, 1, 4, 1), np.uint16), v_cache_bits=np.zeros((3, 1, 4, 1), np.uint16))
    kc_, _, sk, _ = kc.kv_conv_write(**case)
    got = kc.bf16_bits_to_f64(kc_)
    # positions 4, 5, 6: position 4 -> page bt[1] = 0 slot 0; 5, 6 -> page 0 slots 1, 2
    assert got[0, 0, 0, 0] == 54 and got[0, 0, 1, 0] == 30 and got[0, 0, 2, 0] == 17
    assert np.array_equal(kc.bf16_bits_to_f64(sk[0, :, 0, 0]), [2, 3])


def test_agrees_with_numpy_convolution_on_integer_data():
    rng = np.random.default_rng(7)
    case = make_case(rng, ks=4, integer=True)
    kc_, vc_, _, _ = kc.kv_conv_write(**case)
    P = case["page_size"]
    for cache_out, xb, sb, w in ((kc_, case["k_new_bits"], case["state_k_bits"], case["w_k"]),
                                 (vc_, case["v_new_bits"], case["state_v_bits"], case["w_v"])):
        for b in range(3):
            t0, t1 = case["cu_q"][b], case["cu_q"][b + 1]
            n, L = t1 - t0, case["seq_lens"][b]
            hist = kc.bf16_bits_to_f64(np.concatenate([sb[b], xb[t0:t1]], axis=0))
            for g in range(hist.shape[1]):
                for d in range(hist.shape[2]):
                    full = np.convolve(hist[:, g, d], w[g, d, ::-1], mode="valid")   # causal taps
                    for i in range(n):
                        p = L - n + i
                        pg = case["block_table"][b][p // P]
                        assert kc.bf16_bits_to_f64(cache_out[pg, g, p % P, d]) == full[i]


def test_two_steps_with_the_carried_state_equal_one_step():
    check_two_steps(kc)


def check_two_steps(kc):
    rng = np.random.default_rng(11)
    ks = 4
    whole = make_case(rng, ks=ks, n=(6, 4, 7), L=(6, 9, 12))
    kc_w, vc_w, sk_w, sv_w = kc.kv_conv_write(**whole)
    # the same tokens in two steps: first m of each request, then the rest
    m = (2, 1, 5)
    n = (6, 4, 7)
    cu = whole["cu_q"]
    idx1 = np.concatenate([np.arange(cu[b], cu[b] + m[b]) for b in range(3)])
    idx2 = np.concatenate([np.arange(cu[b] + m[b], cu[b + 1]) for b in range(3)])
    step1 = dict(whole, k_new_bits=whole["k_new_bits"][idx1], v_new_bits=whole["v_new_bits"][idx1],
                 cu_q=np.concatenate([[0], np.cumsum(m)]).astype(np.int32),
                 seq_lens=np.array([whole["seq_lens"][b] - n[b] + m[b] for b in range(3)], np.int32))
    k1, v1, sk1, sv1 = kc.kv_conv_write(**step1)
    step2 = dict(whole, k_new_bits=whole["k_new_bits"][idx2], v_new_bits=whole["v_new_bits"][idx2],
                 cu_q=np.concatenate([[0], np.cumsum([n[b] - m[b] for b in range(3)])]).astype(np.int32),
                 state_k_bits=sk1, state_v_bits=sv1, k_cache_bits=k1, v_cache_bits=v1)
    k2, v2, sk2, sv2 = kc.kv_conv_write(**step2)
    assert np.array_equal(k2, kc_w) and np.array_equal(v2, vc_w)
    assert np.array_equal(sk2, sk_w) and np.array_equal(sv2, sv_w)


def test_magnitude_bounds_the_value_and_is_tight_without_cancellation():
    """mag = sum_j |w_j x_j| is >= |y| always, and == |y| when every term has one sign."""
    rng = np.random.default_rng(21)
    case = make_case(rng, ks=4)
    y, mag, page, slot, _ = kc.kv_conv_rows(x_bits=case["k_new_bits"], cu_q=case["cu_q"],
                                            seq_lens=case["seq_lens"], block_table=case["block_table"],
                                            page_size=case["page_size"], w=case["w_k"], ks=4,
                                            state_bits=case["state_k_bits"])
    assert (mag >= np.abs(y) - 1e-12).all() and (mag > 0).any()
    pos = dict(case)
    pos["k_new_bits"] = to_bits(np.abs(kc.bf16_bits_to_f64(case["k_new_bits"])))
    pos["state_k_bits"] = to_bits(np.abs(kc.bf16_bits_to_f64(case["state_k_bits"])))
    y2, mag2, *_ = kc.kv_conv_rows(x_bits=pos["k_new_bits"], cu_q=case["cu_q"], seq_lens=case["seq_lens"],
                                   block_table=case["block_table"], page_size=case["page_size"],
                                   w=np.abs(case["w_k"]), ks=4, state_bits=pos["state_k_bits"])
    assert np.allclose(mag2, y2, rtol=1e-15, atol=0)
    # rows map to the slots of their positions; rows of no request (none here) would be -1
    assert (page >= 0).all() and ((0 <= slot) & (slot < case["page_size"])).all()


def test_mutants_fail_the_pins():
    """Plausible mistakes planted in copies of the oracle must each fail a pin."""
    import importlib.util, pathlib
    src = pathlib.Path(kc.__file__).read_text()
    mutants = {
        "reversed taps": ("y += w[:, :, j] * hist[i + j]", "y += w[:, :, ks - 1 - j] * hist[i + j]"),
        "state ignored": ("prev = bf16_bits_to_f64(st_bits[b]) if ks > 1 else np.zeros((0, Hkv, D))",
                          "prev = np.zeros((ks - 1, Hkv, D))"),
        "off-by-one position": ("p = L - n + i\n", "p = L - n + i - 1\n"),
        "stale state": ("axis=0)[n:]", "axis=0)[:ks - 1]"),
    }
    for name, (a, b) in mutants.items():
        assert a in src, name
        spec = importlib.util.spec_from_loader(f"kc_mut_{abs(hash(name))}", loader=None)
        mod = importlib.util.module_from_spec(spec)
        exec(src.replace(a, b), mod.__dict__)
        failed = False
        for check in (lambda: check_one_hot_shift(mod, 3), lambda: check_hand_worked(mod),
                      lambda: check_two_steps(mod)):
            try:
                check()
            except (AssertionError, IndexError, ValueError):
                failed = True
        assert failed, f"mutant '{name}' passed every pin"
