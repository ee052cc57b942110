"""The closed-form scale s_i = (E|X_i|)^alpha / mean_j |W_ij|, CUDA path
against the CPU oracle: bit-exact (both sum the row magnitudes exactly in
fp64 and round one fp64 quotient to fp32)."""
import numpy as np
import pytest
import torch

from gpu_common import custom_cpu, require_gpu, workload_cpu
from oracle import awq_oracle as orc
from post_weight_quantization_column_b300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def awq():
    return require_gpu()


@pytest.mark.parametrize("name", ["tiny", "attn_proj", "mlp_down", "large_mlp"])
@pytest.mark.parametrize("alpha", [0.5, 0.0, 1.0, 0.35])
def test_closed_form_bit_exact(awq, name, alpha):
    w, X, W, Xf, Wf = workload_cpu(name)
    a = orc.act_stats(Xf)       # the oracle's statistic is the input of both sides
    s = awq.closed_form_scales(W.cuda(), torch.from_numpy(a).cuda(), alpha).cpu().numpy()
    assert np.array_equal(s, orc.closed_form_scales(Wf, a, alpha))


def test_closed_form_zero_row_dead_channel_and_pack(awq):
    w = synth.custom("closedform", 61, 128, 384, 264, symmetric=False)
    _, X, W, Xf, Wf = custom_cpu(w)
    Wf = Wf.copy()
    Wf[7] = 0.0                 # a zero row: s = 1
    a = orc.act_stats(Xf)
    a[11] = 0.0                 # a dead channel: the floor
    Wb = synth.to_bf16(Wf)
    s = awq.closed_form_scales(Wb.cuda(), torch.from_numpy(a).cuda()).cpu().numpy()
    want = orc.closed_form_scales(Wf, a)
    assert np.array_equal(s, want) and s[7] == 1.0
    assert s[11] == orc.closed_form_scales(Wf[11:12], np.array([0.0], dtype=np.float32))[0]
    qw, sc, z = awq.quantize_pack(Wb.cuda(), torch.from_numpy(s).cuda(), 128, False)
    oq, osc, oz = orc.pack(Wf, want, 128, False)
    assert np.array_equal(qw.cpu().numpy(), oq)
    assert np.array_equal(sc.cpu().numpy().view(np.uint16), osc.view(np.uint16))
    assert np.array_equal(z.cpu().numpy().view(np.uint16), oz.view(np.uint16))
