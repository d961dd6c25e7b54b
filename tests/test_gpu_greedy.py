"""Greedy (temperature 0) chain and tree verification vs the oracle.
Integer outputs must be bit-exact."""

import numpy as np
import pytest
import torch

import synth
from oracle.chain import verify_chain
from oracle.tree import verify_tree
from tests._parity import compare_chain, compare_tree, lib_ready

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()


def api():
    from speculative_decoding_verification_tree_gb300 import api as a
    return a


def _run_chain(w, dev="cuda"):
    target, _, toks = synth.chain_inputs(w, dev)
    gpu = api().spec_verify_chain(target, None, toks, temperature=0.0)
    torch.cuda.synchronize()
    ref = verify_chain(target.cpu().float().numpy(), None, toks.cpu().numpy(),
                       temperature=0.0)
    return gpu, ref


@pytest.mark.parametrize("V,dtype", [(1, torch.bfloat16), (37, torch.float32),
                                     (1000, torch.bfloat16),
                                     (16384 * 2 + 8, torch.bfloat16),
                                     (40001, torch.float32),
                                     (50000, torch.bfloat16)])
def test_greedy_chain_small(V, dtype):
    w = synth.workload("greedy", B=7, K=5, V=V, target_dtype=dtype)
    gpu, ref = _run_chain(w)
    compare_chain(gpu, ref, greedy=True)


def test_greedy_chain_k1_b1_and_k0():
    w = synth.workload("greedy", B=1, K=1, V=333)
    gpu, ref = _run_chain(w)
    compare_chain(gpu, ref, greedy=True)
    w = synth.workload("greedy", B=3, K=0, V=333)
    gpu, ref = _run_chain(w)
    compare_chain(gpu, ref, greedy=True, check_mass=False)


def test_greedy_ties_nan_inf():
    dev = "cuda"
    B, K, V = 4, 3, 3000
    t = torch.zeros(B, K + 1, V)
    t[0, :, 5] = 1.0
    t[0, :, 9] = 1.0              # exact tie: index 5 wins
    t[1] = float("-inf")          # all -inf: index 0
    t[2, :, :] = float("nan")
    t[2, :, 17] = 3.0             # NaN ignored
    t[3] = torch.randint(-2, 3, (K + 1, V)).float()  # many ties
    tb = t.to(torch.bfloat16).to(dev)
    toks = torch.tensor([[5, 5, 9], [0, 0, 1], [17, 17, 17], [0, 1, 2]],
                        dtype=torch.int32, device=dev)
    gpu = api().spec_verify_chain(tb, None, toks, temperature=0.0)
    ref = verify_chain(tb.cpu().float().numpy(), None, toks.cpu().numpy(),
                       temperature=0.0)
    compare_chain(gpu, ref, greedy=True)


def test_greedy_full_size_workload():
    # B=256, K=8, V=128256 bf16, the configuration bench.py times
    w = synth.workload("greedy")
    gpu, ref = _run_chain(w)
    compare_chain(gpu, ref, greedy=True)
    acc = gpu[0].cpu().numpy()
    assert 0 < acc.mean() < 8  # roughly half the drafts are accepted


def test_greedy_tree_matches_oracle():
    w = synth.workload("tree_static", B=6, V=3000, temperature=0.0)
    target, _, _, toks, par = synth.tree_inputs(w, "cuda")
    # make some children hit the argmax of their parent row
    am = target.float().argmax(-1)
    pl = par[0].tolist()
    for j in range(len(pl)):
        if j % 3 == 0:
            toks[:, j] = am[:, pl[j] + 1].to(torch.int32)
    gpu = api().spec_verify_tree(target, None, None, toks, par,
                                 temperature=0.0)
    ref = verify_tree(target.cpu().float().numpy(), None,
                      np.full((6, 61), -1), toks.cpu().numpy(),
                      par.cpu().numpy(), temperature=0.0)
    compare_tree(gpu, ref, greedy=True)
    assert ref.path_len.max() >= 1
