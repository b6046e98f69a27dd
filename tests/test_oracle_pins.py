"""Pins for the fp64 oracle: it must agree with things other than itself.

Nothing on the pages prints a worked attention value, so the oracle is pinned by
(1) a second, materialised-matrix restatement on tiny inputs (brute force), (2) closed
forms, (3) reduction to a library routine (PyTorch scaled-dot-product attention with
an explicit bottom-right causal mask), (4) invariances the definition implies, (5) exact
bookkeeping probes, (6) a hand-worked golden file, and (7) bug re-injection: mutants of
the oracle source must fail these pins.

Definition followed: "Support Inkling-NVFP4 model" (TensorRT-LLM PR #17062), section
"Architecture" (pre-softmax bias per query token, head and distance; 512-key windows,
full-causal global layers); GQA map and positional paging from "Inkling attn backend
cleanup fake registry" (TensorRT-LLM PR #17860).
"""
import json
import math
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from paged_attention_relative_gqa_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def run_oracle(prob, lib=None):
    return oracle.attention(**prob.oracle_kwargs(), lib=lib) if lib else oracle.attention(**prob.oracle_kwargs())


def run_brute(prob):
    return brute.attention(**prob.oracle_kwargs())


def random_tiny(rng, seed):
    G = int(rng.choice([1, 2, 4, 8]))
    Hkv = int(rng.choice([1, 2]))
    P = int(rng.choice([1, 2, 4, 16]))
    Wn = int(rng.choice([-1, 1, 3, 7]))
    E = int(rng.choice([1, 4, 64]))
    D = int(rng.choice([4, 8, 16]))
    B = int(rng.integers(1, 4))
    Ls, ns = [], []
    for _ in range(B):
        L = int(rng.integers(0, 41))
        n = 0 if L == 0 else int(rng.integers(1, L + 1))
        Ls.append(L)
        ns.append(n)
    scale = float(rng.choice([1.0 / math.sqrt(D), 1.0 / D, 0.7]))
    return W.make_problem(num_q_heads=G * Hkv, num_kv_heads=Hkv, head_dim=D, page_size=P,
                          rel_extent=E, window=Wn, q_lens=ns, seq_lens=Ls, seed=seed,
                          sm_scale=scale, max_pages=max([-(-L // P) for L in Ls] + [1]) + 2)


# ---------------------------------------------------------------- (1) brute force

def test_oracle_matches_brute_force_on_tiny_cases():
    rng = np.random.default_rng(1234)
    rows = 0
    for case in range(240):
        prob = random_tiny(rng, seed=case)
        a = run_oracle(prob)
        b = run_brute(prob)
        assert np.all(np.isfinite(a))
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12, err_msg=f"case {case}")
        rows += a.shape[0] * a.shape[1]
    print(f"brute-force pin: {rows} rows compared")
    assert rows > 1000


# ---------------------------------------------------------------- (2) closed forms

def _single(L, n=1, **kw):
    base = dict(num_q_heads=1, num_kv_heads=1, head_dim=8, page_size=4, rel_extent=64,
                window=-1, q_lens=[n], seq_lens=[L], seed=7)
    base.update(kw)
    return W.make_problem(**base)


def _v_row(prob, b, k, g=0):
    pg = int(prob.block_table[b, k // prob.page_size])
    return prob.v_cache[pg, g, k % prob.page_size].float().double().numpy()


def test_closed_form_single_key_returns_its_value():
    prob = _single(1)
    out = run_oracle(prob)
    np.testing.assert_array_equal(out[0, 0], _v_row(prob, 0, 0))


def test_closed_form_two_keys_weight_is_logistic_of_bias_gap():
    prob = _single(2)
    # zero keys so only the bias separates the two scores
    prob.k_cache.zero_()
    rel = prob.rel_logits
    rel[0, 0, 0] = 0.9   # distance 0: key 1 (the token itself)
    rel[0, 0, 1] = -0.4  # distance 1: key 0
    out = run_oracle(prob)[0, 0]
    w1 = 1.0 / (1.0 + math.exp(-(float(np.float32(0.9)) - float(np.float32(-0.4)))))
    expect = w1 * _v_row(prob, 0, 1) + (1 - w1) * _v_row(prob, 0, 0)
    np.testing.assert_allclose(out, expect, rtol=0, atol=1e-14)


def test_closed_form_window_one_returns_own_value():
    prob = _single(13, n=13, window=1)
    out = run_oracle(prob)
    for i in range(13):
        np.testing.assert_array_equal(out[i, 0], _v_row(prob, 0, i))


# ---------------------------------------------------------------- (3) library routine

@pytest.mark.parametrize("window", [-1, 0, 64])
def test_reduces_to_causal_sdpa_when_bias_is_zero(window):
    G, Hkv, D, P, L, n = 2, 2, 16, 4, 37, 11
    prob = W.make_problem(num_q_heads=G * Hkv, num_kv_heads=Hkv, head_dim=D, page_size=P,
                          rel_extent=8, window=window, q_lens=[n], seq_lens=[L], seed=3)
    prob.rel_logits.zero_()
    out = run_oracle(prob)
    # logical K/V history through the table, then PyTorch SDPA in fp64
    npg = -(-L // P)
    pages = prob.block_table[0, :npg].long()
    K = prob.k_cache[pages].double().permute(0, 2, 1, 3).reshape(npg * P, Hkv, D)[:L]
    V = prob.v_cache[pages].double().permute(0, 2, 1, 3).reshape(npg * P, Hkv, D)[:L]
    K = K.repeat_interleave(G, dim=1).permute(1, 0, 2)  # [Hq, L, D]
    V = V.repeat_interleave(G, dim=1).permute(1, 0, 2)
    Q = prob.q.double().permute(1, 0, 2)                 # [Hq, n, D]
    # bottom-right aligned causal mask: query i sits at position L - n + i
    qpos = torch.arange(L - n, L)[:, None]
    mask = torch.arange(L)[None, :] <= qpos
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask,
                                                           scale=prob.sm_scale)
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- (4) invariances

def _prob(seed=11, **kw):
    base = dict(num_q_heads=8, num_kv_heads=2, head_dim=16, page_size=4, rel_extent=16,
                window=9, q_lens=[5, 1, 12], seq_lens=[23, 30, 12], seed=seed)
    base.update(kw)
    return W.make_problem(**base)


def test_row_shift_of_bias_leaves_output_unchanged():
    prob = _prob()
    a = run_oracle(prob)
    c = torch.randn(prob.total_q, prob.num_q_heads, 1, dtype=torch.float32) * 3
    prob.rel_logits += c
    b = run_oracle(prob)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-6)  # bias is fp32: the shift rounds


def test_exact_masking_outside_window_and_past_length():
    prob = _prob()
    a = run_oracle(prob)
    P = prob.page_size
    for b, (n, L) in enumerate(zip(prob.q_lens, prob.seq_lens_list)):
        lo = max(0, L - n - prob.window + 1)   # smallest key any new row of b sees
        for k in range(0, lo):
            pg = int(prob.block_table[b, k // P])
            if lo // P == k // P:               # same page as a visible key: finite junk
                prob.k_cache[pg, :, k % P] = 1e4
                prob.v_cache[pg, :, k % P] = -1e4
            else:                               # wholly invisible page: NaN
                prob.k_cache[pg] = float("nan")
                prob.v_cache[pg] = float("nan")
        npg = -(-L // P)
        for k in range(L, npg * P):             # slots past the length in the last page
            pg = int(prob.block_table[b, k // P])
            prob.v_cache[pg, :, k % P] = 1e4
    # bias buckets no visible key uses: those >= the largest visible distance + 1
    for b, (n, L) in enumerate(zip(prob.q_lens, prob.seq_lens_list)):
        t0 = int(prob.cu_q_lens[b])
        for i in range(n):
            p = L - n + i
            far = min(p, prob.window - 1) + 1
            prob.rel_logits[t0 + i, :, far:] = 1e6
    b = run_oracle(prob)
    assert np.array_equal(a, b)


def test_page_permutation_and_unused_nan_pages_leave_output_bitwise_equal():
    prob = _prob()
    a = run_oracle(prob)
    g = torch.Generator().manual_seed(5)
    extra = 6
    N = prob.num_pages
    perm = torch.randperm(N + extra, generator=g)     # new physical slot of old page i is perm[i]
    shape = (N + extra,) + tuple(prob.k_cache.shape[1:])
    k2 = torch.full(shape, float("nan"), dtype=torch.bfloat16)
    v2 = torch.full(shape, float("nan"), dtype=torch.bfloat16)
    k2[perm[:N]] = prob.k_cache
    v2[perm[:N]] = prob.v_cache
    bt = prob.block_table.clone()
    valid = bt < N
    bt[valid] = perm[bt[valid].long()].to(torch.int32)
    prob.k_cache, prob.v_cache, prob.block_table = k2, v2, bt
    b = run_oracle(prob)
    assert np.array_equal(a, b)


def test_clamp_matches_explicitly_expanded_bias_table():
    E = 5
    prob = _prob(window=-1, rel_extent=E)
    a = run_oracle(prob)
    Lmax = max(prob.seq_lens_list)
    idx = torch.clamp(torch.arange(Lmax), max=E - 1)
    prob.rel_logits = prob.rel_logits[:, :, idx].contiguous()
    prob.rel_extent = Lmax
    b = run_oracle(prob)
    assert np.array_equal(a, b)


def test_gqa_equals_mha_with_repeated_kv():
    prob = _prob()
    a = run_oracle(prob)
    G = prob.num_q_heads // prob.num_kv_heads
    prob.k_cache = prob.k_cache.repeat_interleave(G, dim=1).contiguous()
    prob.v_cache = prob.v_cache.repeat_interleave(G, dim=1).contiguous()
    prob.num_kv_heads = prob.num_q_heads
    b = run_oracle(prob)
    assert np.array_equal(a, b)


def test_decode_equals_last_row_of_prefill():
    prob = _prob(q_lens=[17], seq_lens=[17], window=6)
    pre = run_oracle(prob)
    for p in [0, 3, 5, 6, 16]:
        dec = W.make_problem(num_q_heads=8, num_kv_heads=2, head_dim=16, page_size=4,
                             rel_extent=16, window=6, q_lens=[1], seq_lens=[p + 1], seed=1)
        npg = -(-(p + 1) // 4)
        dec.k_cache, dec.v_cache = prob.k_cache, prob.v_cache
        dec.block_table = prob.block_table[:, :npg].clone()
        dec.q = prob.q[p:p + 1].clone()
        dec.rel_logits = prob.rel_logits[p:p + 1].clone()
        d = run_oracle(dec)
        assert np.array_equal(d[0], pre[p])


# ---------------------------------------------------------------- (5) bookkeeping probes

def _probe_problem(L, n, window, E, P=4, seed=2):
    prob = W.make_problem(num_q_heads=2, num_kv_heads=1, head_dim=8, page_size=P,
                          rel_extent=E, window=window, q_lens=[n], seq_lens=[L], seed=seed)
    prob.q.zero_()
    # V[k, 0:2] = (k // 256, k % 256): exact in bf16
    for k in range(L):
        pg = int(prob.block_table[0, k // P])
        prob.v_cache[pg, 0, k % P, 0] = k // 256
        prob.v_cache[pg, 0, k % P, 1] = k % 256
    return prob


@pytest.mark.parametrize("window,E", [(-1, 64), (7, 16), (1, 4)])
def test_argmax_probe_finds_the_key_at_the_chosen_distance(window, E):
    L, n = 40, 40
    prob = _probe_problem(L, n, window, E)
    rng = np.random.default_rng(0)
    jstar = rng.integers(0, E, size=n)
    prob.rel_logits.fill_(-30.0)
    for i in range(n):
        prob.rel_logits[i, :, jstar[i]] = 30.0
    out = run_oracle(prob)
    for i in range(n):
        p = i
        lo = 0 if window <= 0 else max(0, p - window + 1)
        vis = list(range(lo, p + 1))
        favoured = [k for k in vis if min(p - k, E - 1) == jstar[i]]
        if len(favoured) == 1:
            k = favoured[0]
            got = round(out[i, 0, 0]) * 256 + round(out[i, 0, 1])
            assert got == k, (i, got, k)


def test_count_probe_recovers_number_of_visible_keys():
    for window in (-1, 5, 12):
        L = n = 30
        prob = _probe_problem(L, n, window, E=64)
        prob.rel_logits.zero_()
        for i in range(n):
            lo = 0 if window <= 0 else max(0, i - window + 1)
            for k in range(L):
                pg = int(prob.block_table[0, k // 4])
                prob.v_cache[pg, 0, k % 4, 0] = 1.0
                prob.v_cache[pg, 0, k % 4, 1] = 0.0
            pg = int(prob.block_table[0, lo // 4])
            prob.v_cache[pg, 0, lo % 4, 1] = 1.0
            out = run_oracle(prob)
            count = round(1.0 / out[i, 0, 1])
            expect = i - lo + 1
            assert count == expect
            assert out[i, 0, 0] == pytest.approx(1.0, abs=1e-14)


# ---------------------------------------------------------------- (6) hand-worked golden file

def test_hand_worked_golden_cases():
    with open(os.path.join(GOLDEN, "hand_worked.json")) as f:
        cases = json.load(f)["cases"]
    assert len(cases) >= 3
    for c in cases:
        L, D = c["L"], c["D"]
        prob = W.make_problem(num_q_heads=1, num_kv_heads=1, head_dim=D, page_size=c["P"],
                              rel_extent=c["E"], window=c["window"], q_lens=[1], seq_lens=[L],
                              seed=0, sm_scale=1.0)
        prob.q.zero_()
        P = c["P"]
        for k in range(L):
            pg = int(prob.block_table[0, k // P])
            prob.k_cache[pg, 0, k % P] = 0
            prob.v_cache[pg, 0, k % P] = torch.tensor(c["V"][k], dtype=torch.bfloat16)
        prob.rel_logits[0, 0, :] = torch.tensor(c["bias"], dtype=torch.float32)
        out = run_oracle(prob)[0, 0]
        np.testing.assert_allclose(out, c["expect"], rtol=1e-6, atol=1e-6, err_msg=c["name"])


# ---------------------------------------------------------------- error paths

def test_oracle_rejects_out_of_range_page_for_visible_key():
    prob = _prob()
    L = prob.seq_lens_list[0]
    prob.block_table[0, (L - 1) // prob.page_size] = prob.num_pages + 100
    with pytest.raises(ValueError):
        run_oracle(prob)
    # a page the window never reaches may hold anything: no error
    prob = _prob()
    prob.block_table[0, 0] = prob.num_pages + 100
    run_oracle(prob)


def test_oracle_rejects_more_new_tokens_than_history():
    prob = _prob()
    kw = prob.oracle_kwargs()
    kw["seq_lens"] = kw["seq_lens"].copy()
    kw["seq_lens"][0] = 2
    with pytest.raises(ValueError):
        oracle.attention(**kw)


def test_zero_length_sequence_gives_zero_rows():
    prob = _prob(q_lens=[0, 1, 3], seq_lens=[0, 9, 3])
    out = run_oracle(prob)
    assert out.shape[0] == 4 and np.all(np.isfinite(out))


# ---------------------------------------------------------------- (7) bug re-injection

MUTANTS = {
    "window_one_too_wide": ("p - (window - 1) > 0) lo = p - (window - 1)", "p - window > 0) lo = p - window"),
    "clamp_one_short": ("dist = rel_extent - 1;", "dist = rel_extent > 1 ? rel_extent - 2 : 0;"),
    "gqa_modulo_map": ("const int g = h / group;", "const int g = h % num_kv_heads;"),
    "bias_scaled": ("sm_scale * dot + (double)brow[dist]", "sm_scale * (dot + (double)brow[dist])"),
    "top_left_positions": ("const int64_t p = L - n_b + (t - cu_q[b]);", "const int64_t p = (t - cu_q[b]);"),
    "slot_shift": ("const int64_t slot = k % page_size;\n                const uint16_t* krow",
                   "const int64_t slot = (k + 1) % page_size;\n                const uint16_t* krow"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_reinjected_bug(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc missing")
    old, new = MUTANTS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "attn_ref.c")).read()
    assert old in src, f"mutation target for {name} not found: pin would be vacuous"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new, 1))
    lib = oracle.load(oracle.build(str(mpath), str(tmp_path / "libmutant.so")))
    rng = np.random.default_rng(99)
    caught = False
    for case in range(120):
        prob = random_tiny(rng, seed=case)
        try:
            a = run_oracle(prob, lib=lib)
        except ValueError:
            caught = True
            break
        if not np.allclose(a, run_brute(prob), rtol=0, atol=1e-9):
            caught = True
            break
    assert caught, f"mutant {name} survived the brute-force pin"


# ---------------------------------------------------------------- (8) the sampled-row path
#
# Parity on the large workloads calls ``attention_rows`` with only the sampled rows'
# query vectors and bias rows (``q_rows_bits`` / ``rel_rows``) and placeholders for the
# whole tensors.  That path must give, row for row and bit for bit, what the full-tensor
# path gives; and it must never read the whole tensors when the rows are supplied.

def _rows_path(prob, rng, lib=None):
    """Oracle on a random (t, h) subset through the gathered-rows path.  The gathered rows
    sit at the front of buffers padded with NaN, so a path that indexes them wrongly
    (by packed row instead of sampled row, or with another row stride) reads NaN or other
    rows instead of faulting; the whole q / rel tensors are NaN placeholders."""
    kw = prob.oracle_kwargs()
    q_bits, rel = kw["q_bits"], kw["rel"]
    total_q, Hq, D = q_bits.shape
    E = rel.shape[2]
    n_all = total_q * Hq
    n = int(rng.integers(1, n_all + 1))
    pick = np.sort(rng.choice(n_all, size=n, replace=False))
    rows_t = (pick // Hq).astype(np.int32)
    rows_h = (pick % Hq).astype(np.int32)
    pad = n + total_q + 1
    q_big = np.full((pad * max(1, -(-E // D)), D), 0x7FC0, dtype=np.uint16)   # bf16 NaN
    rel_big = np.full((pad, E), np.nan, dtype=np.float32)
    q_big[:n] = q_bits[rows_t, rows_h]
    rel_big[:n] = rel[rows_t, rows_h]
    kw["q_bits"] = np.full_like(q_bits, 0x7FC0)
    kw["rel"] = np.full_like(rel, np.nan)
    extra = {"lib": lib} if lib is not None else {}
    out = oracle.attention_rows(rows_t=rows_t, rows_h=rows_h, q_rows_bits=q_big[:n],
                                rel_rows=rel_big[:n], **kw, **extra)
    return rows_t, rows_h, out


def test_sampled_rows_path_equals_full_path_bitwise():
    rng = np.random.default_rng(2024)
    rows = 0
    for case in range(200):
        prob = random_tiny(rng, seed=500 + case)
        if int(prob.cu_q_lens[-1]) == 0:
            continue
        full = run_oracle(prob)
        t, h, part = _rows_path(prob, rng)
        np.testing.assert_array_equal(part, full[t, h], err_msg=f"case {case}")
        # and against the independent restatement
        np.testing.assert_allclose(part, run_brute(prob)[t, h], rtol=0, atol=1e-12)
        rows += part.shape[0]
    print(f"sampled-row path: {rows} rows compared bit for bit")
    assert rows > 1000


ROW_MUTANTS = {
    "q_rows_by_packed_row": ("q_rows ? q_rows + r * (int64_t)head_dim", "q_rows ? q_rows + t * (int64_t)head_dim"),
    "rel_rows_by_packed_row": ("rel_rows ? rel_rows + r * (int64_t)rel_extent",
                               "rel_rows ? rel_rows + t * (int64_t)rel_extent"),
    "q_rows_stride_E": ("q_rows ? q_rows + r * (int64_t)head_dim", "q_rows ? q_rows + r * (int64_t)rel_extent"),
    "rel_rows_stride_D": ("rel_rows ? rel_rows + r * (int64_t)rel_extent",
                          "rel_rows ? rel_rows + r * (int64_t)head_dim"),
}


@pytest.mark.parametrize("name", sorted(ROW_MUTANTS))
def test_rows_path_pin_catches_reinjected_bug(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc missing")
    old, new = ROW_MUTANTS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "attn_ref.c")).read()
    assert old in src, f"mutation target for {name} not found: pin would be vacuous"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new, 1))
    lib = oracle.load(oracle.build(str(mpath), str(tmp_path / "libmutant.so")))
    rng = np.random.default_rng(77)
    caught = False
    for case in range(120):
        prob = random_tiny(rng, seed=900 + case)
        if int(prob.cu_q_lens[-1]) == 0:
            continue
        t, h, part = _rows_path(prob, rng, lib=lib)
        if not np.allclose(part, run_brute(prob)[t, h], rtol=0, atol=1e-9):
            caught = True
            break
    assert caught, f"mutant {name} survived the sampled-row pin"
