"""Decode called with the previous step's lengths (stale metadata).

A serving step writes its new K/V row into the paged cache before attention reads it.  A
decode launched with the lengths of the step before (every L_b one short) must attend over
exactly the first L_b - 1 keys, with the query at position L_b - 2, and never touch the
slot the newer row went into.  The check is the fp64 oracle on the stale lengths, with the
newest slot of every request (its K and V rows, all heads) poisoned with NaN: one read of
it would make that request's rows NaN.  Some lengths put the newest row at slot 0 of a
page of its own, so the stale call must not read that page at all.
(Failure detection, "Inkling attn backend cleanup fake registry", TensorRT-LLM PR #17860:
decode metadata from an earlier step must not be read as if it were current.)
"""
import dataclasses

import pytest
import torch

from paged_attention_relative_gqa_gb300 import binding
from paged_attention_relative_gqa_gb300 import workloads as W
from tests.parity import compare, oracle_full, run_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()
    yield
    torch.cuda.empty_cache()


def stale_lengths(prob):
    """The same problem with every length one short and the newest slot poisoned."""
    P = prob.page_size
    bt = prob.block_table.cpu()
    k, v = prob.k_cache.clone(), prob.v_cache.clone()
    for b, L in enumerate(prob.seq_lens_list):
        page, slot = int(bt[b, (L - 1) // P]), (L - 1) % P
        k[page, :, slot, :] = float("nan")
        v[page, :, slot, :] = float("nan")
    return dataclasses.replace(prob, seq_lens_list=[L - 1 for L in prob.seq_lens_list],
                               seq_lens=prob.seq_lens - 1, k_cache=k, v_cache=v)


# (Hq, Hkv, D, P, E, W, seq_lens): lengths of the form m P + 1 put the newest row alone on a page
CASES = [
    (16, 4, 128, 64, 1024, 512, [65, 129, 2, 600, 1025, 3000, 513, 514]),    # sliding window 512
    (16, 2, 128, 64, 4096, -1, [4097, 65, 7000, 2, 130, 12289]),             # global, E 4096
    (8, 2, 64, 16, 256, 100, [17, 33, 2, 101, 102, 900]),                    # D 64, P 16, W 100
]


@pytest.mark.parametrize("case", CASES, ids=["swa", "global", "d64_p16"])
def test_decode_with_last_steps_lengths_reads_only_those_keys(case):
    hq, hkv, d, p, e, w, lens = case
    prob = W.make_problem(num_q_heads=hq, num_kv_heads=hkv, head_dim=d, page_size=p, rel_extent=e, window=w,
                          q_lens=[1] * len(lens), seq_lens=lens, seed=61 + len(lens), device=DEV)
    old = stale_lengths(prob)
    out, err = run_gpu(old)
    assert err == 0, f"device error {err:#x}"
    compare(out.float().cpu().numpy(), oracle_full(old), f"decode on the previous step's lengths ({case})")
