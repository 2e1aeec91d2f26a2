"""The block step (verifier-input preparation hoisted ahead of the host's
read of the confidence length; three CUDA graphs) against the oracle.

D = 8 drafts through a 2560 -> 2560 "fast" projection (FP8 activations) and 8
verifier rows through a 2560 -> 32000 "critical" projection (int8 path), the
shapes of the role-dependent workload.  For low and high draft confidence,
with and without hoisting: the confidence length and the decision follow the
hybrid rule, the draft outputs are within the FP8 bound, the verifier codes
and the verifier's accumulators are bit-exact, and a step that needs no
verification launches none (its outputs keep their sentinel)."""
import numpy as np
import pytest
import torch

import oracle
from ternary_w2a8_linear_gb300 import build, inputs
from ternary_w2a8_linear_gb300 import linear as L
from gpu_util import assert_f32_close, assert_fp8_within_bound, bf16_bits, bf16_tensor, dev_tensor, fp8_reference

pytestmark = pytest.mark.gpu

D, R, KD, ND, KV, NV = 8, 8, 2560, 2560, 2560, 32000
TAU, M_MIN = 0.9, 4


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    yield L.load()
    assert L.bitmtp_linear_device_error() == 0


@pytest.fixture(scope="module")
def problem():
    rng = np.random.default_rng(8100)
    Td = inputs.ternary(rng, (ND, KD), 0.5)
    Tv = inputs.ternary(rng, (NV, KV), 0.5)
    wd, wv = np.float32(0.021), np.float32(0.034)
    xd = inputs.normal_with_outliers_bf16(rng, (D, KD))
    xv = inputs.normal_with_outliers_bf16(rng, (R, KV))
    return dict(Td=Td, Tv=Tv, wd=wd, wv=wv, xd=xd, xv=xv, pkd=L.pack(dev_tensor(Td)), pkv=L.pack(dev_tensor(Tv)))


def _step(pr, p, hoist):
    from ternary_w2a8_linear_gb300.blockstep import BlockStep
    stream = torch.cuda.Stream()
    draft = dict(pk=pr["pkd"], w_scale=pr["wd"], N=ND, K=KD, x=bf16_tensor(pr["xd"]),
                 y=torch.empty((D, ND), dtype=torch.float32, device="cuda"),
                 p=torch.tensor(p, dtype=torch.float32, device="cuda"))
    verify = dict(pk=pr["pkv"], w_scale=pr["wv"], N=NV, K=KV, x=bf16_tensor(pr["xv"]),
                  y=torch.full((R, NV), float("nan"), dtype=torch.float32, device="cuda"),
                  acc=torch.zeros((R, NV), dtype=torch.int32, device="cuda"))
    bs = BlockStep(draft, verify, TAU, M_MIN, stream)
    # construction runs each part once (before capturing it): sentinels after it
    torch.cuda.synchronize()
    bs.q.fill_(0x55)
    verify["y"].fill_(float("nan"))
    verify["acc"].zero_()
    draft["y"].fill_(float("nan"))
    torch.cuda.synchronize()
    length, verified = bs.run(hoist=hoist)
    stream.synchronize()
    return bs, draft, verify, length, verified


@pytest.mark.parametrize("hoist", [True, False])
def test_low_confidence_verifies(problem, hoist):
    pr = problem
    p = [0.3, 0.97, 0.4, 0.99, 0.99, 0.99, 0.99, 0.99]  # prefix of 2 < m = 4
    bs, draft, verify, length, verified = _step(pr, p, hoist)
    assert (length, verified) == (2, True)
    # the draft: FP8 within its bound
    assert_fp8_within_bound(KD, pr["wd"], draft["y"].cpu().numpy(), None,
                            fp8_reference(pr["Td"], pr["wd"], pr["xd"], True), False)
    # the verifier inputs and the verifier: the int8 path, exact
    q_ref, s_ref, r_ref = oracle.quant_act_bf16(pr["xv"])
    assert np.array_equal(bs.q.cpu().numpy(), q_ref)
    assert np.array_equal(bs.a_scale.cpu().numpy(), s_ref)
    acc_ref = oracle.gemm_acc(pr["Tv"], q_ref)
    assert np.array_equal(verify["acc"].cpu().numpy(), acc_ref)
    assert_f32_close(verify["y"].cpu().numpy(), oracle.dequant(acc_ref, s_ref, pr["wv"]), acc_ref)


@pytest.mark.parametrize("hoist", [True, False])
def test_high_confidence_skips_verification(problem, hoist):
    pr = problem
    p = [0.1, 0.95, 0.93, 0.99, 0.91, 0.2, 0.99, 0.99]  # prefix of 5 >= m = 4
    bs, draft, verify, length, verified = _step(pr, p, hoist)
    assert (length, verified) == (5, False)
    assert torch.isnan(verify["y"]).all()              # no verifier launch
    assert int(verify["acc"].abs().sum()) == 0
    q = bs.q.cpu().numpy()
    if hoist:  # prepared before the decision, used or not
        assert np.array_equal(q, oracle.quant_act_bf16(pr["xv"])[0])
    else:      # never prepared
        assert np.all(q == 0x55)
    assert_fp8_within_bound(KD, pr["wd"], draft["y"].cpu().numpy(), None,
                            fp8_reference(pr["Td"], pr["wd"], pr["xd"], True), False)


def test_hoisted_and_plain_steps_agree_over_repeated_steps(problem):
    pr = problem
    from ternary_w2a8_linear_gb300.blockstep import BlockStep
    stream = torch.cuda.Stream()
    outs = {}
    for hoist in (True, False):
        draft = dict(pk=pr["pkd"], w_scale=pr["wd"], N=ND, K=KD, x=bf16_tensor(pr["xd"]),
                     y=torch.empty((D, ND), dtype=torch.bfloat16, device="cuda"),
                     p=torch.zeros(D, dtype=torch.float32, device="cuda"))
        verify = dict(pk=pr["pkv"], w_scale=pr["wv"], N=NV, K=KV, x=bf16_tensor(pr["xv"]),
                      y=torch.empty((R, NV), dtype=torch.bfloat16, device="cuda"))
        bs = BlockStep(draft, verify, TAU, M_MIN, stream)
        seen = []
        for i, p in enumerate(([0.5, 0.1] + [0.99] * 6, [0.5] + [0.99] * 7, [0.5, 0.95, 0.95, 0.1] + [0.9] * 4)):
            with torch.cuda.stream(stream):
                draft["p"].copy_(torch.tensor(p, dtype=torch.float32), non_blocking=False)
            stream.synchronize()
            seen.append(bs.run(hoist=hoist))
            stream.synchronize()
            if seen[-1][1]:
                outs[(hoist, i)] = bf16_bits(verify["y"])
        assert seen == [(1, True), (8, False), (3, True)]
    for i in (0, 2):
        assert np.array_equal(outs[(True, i)], outs[(False, i)])
