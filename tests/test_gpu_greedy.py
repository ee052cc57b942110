"""The ADR's per-group coordinate greedy, CUDA path against the CPU oracle.

Each decision is an argmin over floating-point sums, so near-ties can go
either way between an fp32 kernel and the fp64 oracle, and one different
decision changes every later one.  The check therefore replays the kernel's
own decisions in the oracle (``follow=``): at every step the kernel's
candidate errors must match the oracle's, and the candidate it chose must be
optimal under the oracle's errors to within the accumulation tolerance
(and never worse than keeping the current scale).  Most decisions must also
equal the oracle's own argmin exactly.

Tolerance: per-column errors are fp32 sums over the group's rows (<= 256
terms), then over 128 columns in fp32, then over column slices in fp64, so
each candidate's error is within ~(256 + 128) * 2^-24 ~ 2.3e-5 of the exact
value relative to its own size; 5e-5 of that size, plus 5e-5 of the group's
smallest candidate error, is used (candidates whose scaled channel takes
over the range can have errors far above the smallest one).  Decisions are
weighed with 5e-5 of the smallest error, the size of the candidates that
compete for it.
"""
import numpy as np
import pytest
import torch

from gpu_common import custom_cpu, require_gpu, workload_cpu
from oracle import awq_oracle as orc
from post_weight_quantization_column_b300 import synth

pytestmark = pytest.mark.gpu

RTOL = 5e-5


@pytest.fixture(scope="module")
def awq():
    return require_gpu()


def check_replay(Wf, a, g, sym, passes, s, trace, errors):
    s_o, tr_o, err_o = orc.greedy_search(Wf, a, group_size=g, symmetric=sym, passes=passes, follow=trace)
    assert np.array_equal(tr_o, trace)
    assert np.array_equal(s_o, s), "final scales are the candidates of the last decisions"
    cand = orc.greedy_candidates()
    D_in = Wf.shape[0]
    agree = 0
    cur = np.full(D_in, 10)
    for p in range(passes):
        for j in range(D_in):
            e_o = err_o[p, j]
            tol = RTOL * e_o.min()
            np.testing.assert_allclose(errors[p, j], e_o, rtol=RTOL, atol=tol)
            k = int(trace[p, j])
            assert e_o[k] <= e_o.min() + tol, (p, j, k, e_o[k], e_o.min())
            assert e_o[k] <= e_o[cur[j]] + tol
            # the oracle's own decision from the same state
            best = cur[j]
            for c in range(len(cand)):
                if e_o[c] < e_o[best]:
                    best = c
            agree += int(best == k)
            cur[j] = k
    return agree / (passes * D_in)


CASES = [
    # seed, N, D_in, D_out, group, symmetric, passes
    (51, 96, 128, 136, 64, False, 3),
    (52, 64, 256, 96, 128, True, 2),
    (53, 80, 256, 264, 256, False, 1),
]


@pytest.mark.parametrize("seed,N,D_in,D_out,g,sym,passes", CASES,
                         ids=[f"{c[2]}x{c[3]}_g{c[4]}_{'sym' if c[5] else 'asym'}_p{c[6]}" for c in CASES])
def test_greedy_replays_against_oracle(awq, seed, N, D_in, D_out, g, sym, passes):
    w = synth.custom(f"greedy{seed}", seed, N, D_in, D_out, symmetric=sym, group_size=g)
    _, X, W, Xf, Wf = custom_cpu(w)
    a_gpu = awq.act_stats(X.cuda())
    a = a_gpu.cpu().numpy()
    s, tr, er = awq.greedy_search(W.cuda(), a_gpu, group_size=g, symmetric=sym, passes=passes, trace=True,
                                  errors=True)
    agree = check_replay(Wf, a, g, sym, passes, s.cpu().numpy(), tr.cpu().numpy(), er.cpu().numpy())
    assert agree >= 0.9, f"only {agree:.3f} of the decisions equal the oracle's own"
    # the outlier channels end up scaled up
    sal = np.argsort(a)[-max(1, D_in // 100):]
    assert np.all(s.cpu().numpy()[sal] >= 1.0)


def test_greedy_full_size_properties(awq):
    """The attention-projection layer at full size: the kernel's own errors
    never rise, the run is deterministic, and the pack at the greedy's scales
    is bit-exact against the oracle on a column sample."""
    w, X, W, Xf, Wf = workload_cpu("attn_proj")
    Xd, Wd = X.cuda(), W.cuda()
    a = awq.act_stats(Xd)
    s, tr, er = awq.greedy_search(Wd, a, group_size=w.group_size, symmetric=w.symmetric, trace=True, errors=True)
    s2, tr2, er2 = awq.greedy_search(Wd, a, group_size=w.group_size, symmetric=w.symmetric, trace=True, errors=True)
    assert torch.equal(s, s2) and torch.equal(tr, tr2) and torch.equal(er, er2)
    s, tr, er = s.cpu().numpy(), tr.cpu().numpy(), er.cpu().numpy()
    cand = orc.greedy_candidates()
    assert np.array_equal(s, cand[tr[-1]])
    cur = np.full(w.D_in, 10)
    for p in range(tr.shape[0]):
        e = er[p, np.arange(w.D_in), :]
        chosen = e[np.arange(w.D_in), tr[p]]
        stay = e[np.arange(w.D_in), cur]
        assert np.all(chosen <= stay * (1 + 1e-9))
        assert np.all(chosen <= e.min(axis=1) * (1 + RTOL))
        cur = tr[p]
    sd = torch.from_numpy(s).cuda()
    qw, sc, z = awq.quantize_pack(Wd, sd, w.group_size, w.symmetric)
    cols = synth.sample_columns(w.D_out, 512, w.seed)
    oq, osc, oz = orc.pack(Wf[:, cols], s, w.group_size, w.symmetric)
    assert np.array_equal(qw[:, cols].cpu().numpy(), oq)
    assert np.array_equal(sc[:, cols].cpu().numpy().view(np.uint16), osc.view(np.uint16))


@pytest.mark.parametrize("sym", [False, True], ids=["asym", "sym"])
def test_greedy_subnormal_step_group(awq, sym):
    """A group so small that its fp16 step is subnormal and rounds far down:
    asymmetric, a negative group whose zero is clamped at 15; symmetric, a
    group whose largest |w'|/step exceeds 7.5.  Codes there need the clamps
    of the exact form; the kernel's decisions replay against the oracle."""
    rng = np.random.default_rng(23)
    D_in, D_out = 256, 64
    Wf = (rng.standard_normal((D_in, D_out)) * 0.02).astype(np.float32)
    m = np.float32((21.0 if not sym else 9.8) * 2.0 ** -24)
    frac = rng.random((128, D_out)).astype(np.float32)
    Wf[:128] = -frac * m if not sym else (frac * 2 - 1) * m
    Wf[0] = -m
    Wb = synth.to_bf16(Wf)
    Wf = synth.bf16_to_f32(Wb)
    a = (rng.random(D_in) + 0.1).astype(np.float32)
    s, tr, er = awq.greedy_search(Wb.cuda(), torch.from_numpy(a).cuda(), group_size=128, symmetric=sym, passes=1,
                                  trace=True, errors=True)
    check_replay(Wf, a, 128, sym, 1, s.cpu().numpy(), tr.cpu().numpy(), er.cpu().numpy())
