"""Parity of the decode layer (projections + absorbed attention, through the C ABI)
with the oracle's plain layer ([N1] forward_decode) in fp64.

The GPU path rounds five intermediates to bf16 that the oracle keeps in fp64
(c^Q, q^C, q^R, the per-head output O, and the layer output), each about 2^-9
relative; through the random projections these add up to a few 1e-3 relative.
Tolerance: relative L2 1e-2 on the layer output y and on O.  The cache rows of
the new tokens are the bf16 rows the format stores on both sides.
"""

import numpy as np
import pytest
import torch

from oracle import mla_oracle as O
from mla_absorbed_decode_absorb_gb300 import workloads as W
from test_gpu_parity import bits, rel_l2

pytestmark = pytest.mark.gpu

Y_REL_L2 = 1e-2


def f64(t):
    return O.bf16_bits_to_f64(bits(t))


def oracle_layer(li, b):
    inp = li.base
    hc, hk = inp.history(b)
    L = int(inp.prior_lens[b])
    kr_hist = O.bf16_bits_to_f64(O.rope_key_bf16_bits(bits(hk), np.arange(L))) if L else np.zeros((0, 64))
    return O.decode_layer(f64(li.x[b]), f64(li.w_dkv), f64(li.w_kr), f64(li.w_dq), f64(li.w_uq), f64(li.w_qr),
                          f64(inp.w_uk), f64(inp.w_uv), f64(li.w_o), f64(hc) if L else np.zeros((0, 512)),
                          kr_hist, L)


def run_layer(li, **kw):
    from mla_absorbed_decode_absorb_gb300 import ops
    from mla_absorbed_decode_absorb_gb300.runtime import LayerSession
    s = LayerSession(li, **kw)
    s.step()
    torch.cuda.synchronize()
    assert ops.mla_get_device_status() == ops.MLA_OK
    return s


def check_layer(s, li, seqs):
    y = s.y.float().cpu().numpy().reshape(li.workload.batch, li.workload.n_q, -1)
    o = s.dec.out.float().cpu().numpy()
    ys, yr, os_, or_ = [], [], [], []
    for b in seqs:
        y_ref, o_ref = oracle_layer(li, b)
        ys.append(y[b]), yr.append(y_ref), os_.append(o[b]), or_.append(o_ref)
    assert rel_l2(np.concatenate(os_), np.concatenate(or_)) <= Y_REL_L2, rel_l2(np.concatenate(os_), np.concatenate(or_))
    assert rel_l2(np.concatenate(ys), np.concatenate(yr)) <= Y_REL_L2, rel_l2(np.concatenate(ys), np.concatenate(yr))


SMALL = {
    "edges": W.Workload("layer_edges", batch=4, n_q=1, lengths=(0, 63, 64, 300), d_model=W.D_MODEL),
    "mtp": W.Workload("layer_mtp", batch=2, n_q=3, lengths=(5, 130), d_model=W.D_MODEL),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_layer_parity_small(name):
    li = W.generate_layer(SMALL[name], seed=5)
    s = run_layer(li)
    check_layer(s, li, range(li.workload.batch))


def test_layer_full_size_sampled():
    """The layer benchmark workload at full size, in the bench's launch configuration;
    the oracle checks the first and the last sequence."""
    li = W.generate_layer(W.LAYER_WORKLOADS["layer_b32_l4096"], seed=0)
    s = run_layer(li)
    check_layer(s, li, [0, li.workload.batch - 1])


@pytest.mark.parametrize("name", sorted(SMALL))
def test_layer_fold_parity_small(name):
    """The weight pre-folds (W_UK^T W_UQ into the query, W_O W_UV into the output) give
    the same layer: one more bf16 rounding (of the folded weights and of O') than the
    unfolded path, the same tolerance."""
    li = W.generate_layer(SMALL[name], seed=6)
    s = run_layer(li, fold=True)
    y = s.y.float().cpu().numpy().reshape(li.workload.batch, li.workload.n_q, -1)
    ys, yr = [], []
    for b in range(li.workload.batch):
        y_ref, _ = oracle_layer(li, b)
        ys.append(y[b]), yr.append(y_ref)
    assert rel_l2(np.concatenate(ys), np.concatenate(yr)) <= Y_REL_L2, rel_l2(np.concatenate(ys), np.concatenate(yr))


def test_layer_fold_full_size_sampled():
    """The folded layer benchmark workload at full size (B = 32, context 4096, the
    1.2 GB of folded weights), in the bench's launch configuration; the oracle
    checks the first and the last sequence."""
    li = W.generate_layer(W.LAYER_WORKLOADS["layer_b32_l4096_fold"], seed=0)
    s = run_layer(li, fold=True)
    y = s.y.float().cpu().numpy().reshape(li.workload.batch, li.workload.n_q, -1)
    ys, yr = [], []
    for b in (0, li.workload.batch - 1):  # the folded path has no per-head O: the layer output is checked
        y_ref, _ = oracle_layer(li, b)
        ys.append(y[b]), yr.append(y_ref)
    err = rel_l2(np.concatenate(ys), np.concatenate(yr))
    print(f"layer_b32_l4096_fold: rel-L2 y {err:.3e}")
    assert err <= Y_REL_L2, err


def test_fold_weights_match_their_definition():
    """W_QK[(h, m), c] = sum_d W_UK[h, d, m] W_UQ[h*128 + d, c] and
    W_OV[j, (h, m)] = sum_d W_O[j, h*128 + d] W_UV[h, d, m], on sampled heads."""
    li = W.generate_layer(SMALL["edges"], seed=7)
    s = run_layer(li, fold=True)
    wqk = s.w_qk.float().cpu().numpy()
    wov = s.w_ov.float().cpu().numpy()
    w_uk, w_uv = f64(li.base.w_uk), f64(li.base.w_uv)
    w_uq, w_o = f64(li.w_uq), f64(li.w_o)
    for h in (0, 77, 127):
        ref_qk = w_uk[h].T @ w_uq[h * 128:(h + 1) * 128]
        ref_ov = w_o[:, h * 128:(h + 1) * 128] @ w_uv[h]
        got_qk = wqk[h * 512:(h + 1) * 512]
        got_ov = wov[:, h * 512:(h + 1) * 512]
        assert np.abs(got_qk - ref_qk).max() <= 2.0 ** -8 * np.abs(ref_qk).max() + 1e-6
        assert np.abs(got_ov - ref_ov).max() <= 2.0 ** -8 * np.abs(ref_ov).max() + 1e-6
