"""The dense towers (ctr_towers_fwd) against the oracle, through the C ABI.

Two references per case, both scaled to the largest logit |y|max:
  * the oracle with every GEMM operand rounded to bf16 as the kernel takes it,
    within 2^-8 |y|max (one bf16 unit of the largest logit). The two differ
    only in accumulation (fp32 on the tensor cores, fp64 in the oracle), and
    where that moves a hidden activation across a bf16 rounding boundary the
    activation changes by one bf16 unit, which the later layers (Xavier
    weights, gain near 1) carry to the logit at about that relative size;
  * the fp64 oracle, within 2^-6 |y|max: each of the four GEMMs rounds both
    operands to bf16 (2^-9 relative each), eight such roundings in all.
"""
import numpy as np
import pytest
import torch

import oracle
from recsys_sparse_embedding_gb300 import binding, synth

from helpers import DeviceRun

pytestmark = pytest.mark.gpu


def run_towers(pooled, din, weights, B=None, prepare=True, device="cuda"):
    B = pooled.shape[0] if B is None else B
    tw = binding.Towers([torch.from_numpy(w) for w in weights], device=device)
    if prepare:
        tw.prepare()
    else:
        tw.buf.zero_()
    p = torch.from_numpy(np.ascontiguousarray(pooled, np.float32)).to(device)
    d = torch.from_numpy(np.ascontiguousarray(din, np.float32)).to(device)
    logit = torch.full((max(B, 1),), float("nan"), device=device)
    st = torch.zeros(1, dtype=torch.int32, device=device)
    binding.ctr_towers_fwd(p, d, B, tw, logit, status=st)
    torch.cuda.synchronize()
    return logit.cpu().numpy()[:B], int(st.item())


def check(pooled, din, weights, name):
    got, st = run_towers(pooled, din, weights)
    assert st == 0, "status 0x%x" % st
    emul = oracle.towers(pooled, din.astype(np.float32), *weights, bf16_mlp=True)
    ref = oracle.towers(pooled, din.astype(np.float32), *weights)
    ymax = float(np.abs(ref).max())
    err_e = np.abs(got - emul).max()
    err = np.abs(got - ref).max()
    print("%s: max|err| vs bf16 oracle %.3e, vs fp64 %.3e; std(ref) %.3e max|ref| %.3e"
          % (name, err_e, err, np.std(ref), ymax))
    assert err_e <= 2.0 ** -8 * ymax, "%s: max err vs bf16 oracle %.3e" % (name, err_e)
    assert err <= 2.0 ** -6 * ymax, "%s: max err vs fp64 oracle %.3e" % (name, err)
    if got.size > 1:  # the logits spread over many tolerance widths
        assert np.std(ref) > 20 * 2.0 ** -8 * ymax


@pytest.mark.parametrize("wl,B,seed", [("taobao", 1000, 3), ("long_multihot", 777, 5)])
def test_towers_on_sparse_path_outputs(wl, B, seed):
    """The CTR forward: din_sparse_fwd, then the towers on its device outputs."""
    batch = synth.generate(wl, seed=seed, B=B, nonzero_bias=True)
    pooled, din, _, st = DeviceRun(batch).fwd(binding.DSF_MODE_BF16_TC, logits=False)
    assert st == 0
    check(pooled, din, synth.tower_weights(seed, bias=0.1), wl)


@pytest.mark.parametrize("B", [1, 127, 128, 129, 300, 4099])
def test_towers_ragged_batches(B):
    """Tile edges: a lone sample, one short tile, exactly one tile, one over,
    and a ragged tail after many tiles."""
    rng = np.random.default_rng(B)
    pooled = (rng.standard_normal((B, 256)) * 0.3).astype(np.float32)
    din = (rng.standard_normal((B, 48)) * 0.05).astype(np.float32)
    check(pooled, din, synth.tower_weights(B, bias=0.2), "B=%d" % B)


def test_towers_large_activations():
    """Inputs of N(0, 4): hidden activations far from 1, so the bf16 rounding
    works on larger exponents and any mis-scaled bias shows."""
    rng = np.random.default_rng(11)
    B = 512
    pooled = (rng.standard_normal((B, 256)) * 4.0).astype(np.float32)
    din = (rng.standard_normal((B, 48)) * 2.0).astype(np.float32)
    w = synth.tower_weights(11, bias=1.0)
    check(pooled, din, w, "N(0, 4) inputs")


def test_towers_not_prepared_sets_the_flag():
    rng = np.random.default_rng(0)
    pooled = rng.standard_normal((200, 256)).astype(np.float32)
    din = rng.standard_normal((200, 48)).astype(np.float32)
    got, st = run_towers(pooled, din, synth.tower_weights(0), prepare=False)
    assert st & binding.FLAG_NOT_PREPARED
    assert np.isnan(got).all()


def test_towers_batch_zero_is_a_no_op():
    got, st = run_towers(np.zeros((0, 256), np.float32), np.zeros((0, 48), np.float32),
                         synth.tower_weights(0))
    assert st == 0 and got.size == 0
