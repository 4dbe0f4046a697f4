"""Verify steps (several tokens per sequence, a state slot per token) through
the C ABI against the CPU oracle, and against the same tokens run as
successive decode steps on the GPU."""
import numpy as np
import pytest
import torch

from gated_deltanet_layer_gb300 import GdnDecode, workloads as WL
from gdn_harness import CORE_COS, CORE_MAX_ABS, STATE_BF16_MAX_ABS, STATE_F32_MAX_ABS, bf16_ulp, cosine, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _inputs(shape, S, T, seed, first_layer=False, pad=()):
    rng = np.random.default_rng(seed)
    w = WL.make_weights(shape, seed)
    st = WL.make_state(shape, seed + 1)
    stp = WL.make_step(shape, S * T, seed + 2, first_layer=first_layer)
    slots = rng.permutation(np.arange(1, shape.num_slots))[:S + S * T]
    sin = slots[:S].astype(np.int32)
    sout = slots[S:].reshape(S, T).astype(np.int32)
    for s in pad:
        sin[s] = 0
    return w, st, stp, sin, sout


def _run_verify(shape, w, st, stp, sin, sout):
    dw = {k: (v.cuda() if v is not None else None) for k, v in w.items()}
    conv, ssm = st["conv_state"].cuda(), st["ssm_state"].cuda()
    layer = GdnDecode(shape)
    core, res = layer.verify(stp["x"].cuda(), stp["residual"].cuda() if stp["residual"] is not None else None, dw,
                             torch.from_numpy(sin).cuda(), torch.from_numpy(sout).cuda(), conv, ssm)
    torch.cuda.synchronize()
    assert layer.check()[0] == 0
    return core, res, conv, ssm


def _compare(shape, w, st, stp, sin, sout, core, res, conv, ssm):
    from oracle import gdn_oracle as O
    ref = O.gdn_verify(shape, f64(stp["x"]), f64(stp["residual"]), {k: f64(v) for k, v in w.items()}, sin, sout,
                       f64(st["conv_state"]), f64(st["ssm_state"]))
    np.testing.assert_array_equal(f64(res), ref["residual_out"])
    S, T = sout.shape
    gcore = f64(core)
    live = [s for s in range(S) if sin[s] > 0]
    for s in range(S):
        if s not in live:
            assert np.all(gcore[s * T:(s + 1) * T] == 0.0)
    rows = [s * T + t for s in live for t in range(T)]
    assert cosine(gcore[rows], ref["core"][rows]) >= CORE_COS
    assert float(np.max(np.abs(gcore[rows] - ref["core"][rows]))) <= CORE_MAX_ABS
    gssm, gconv = f64(ssm), f64(conv)
    written = sorted(int(o) for s in live for o in sout[s])
    others = [i for i in range(shape.num_slots) if i not in written]
    np.testing.assert_array_equal(gssm[others], f64(st["ssm_state"])[others])
    np.testing.assert_array_equal(gconv[others], f64(st["conv_state"])[others])
    tol = STATE_BF16_MAX_ABS if shape.ssm_dtype == "bf16" else STATE_F32_MAX_ABS
    assert float(np.max(np.abs(gssm[written] - ref["ssm_state"][written]))) <= tol
    # conv taps: the kernel's projection values may sit one bf16 ulp from the oracle's
    g, r = gconv[written], ref["conv_state"][written]
    assert np.all(np.abs(g - r) <= bf16_ulp(r) + 2e-3)


@pytest.mark.parametrize("S,T", [(4, 2), (2, 4), (1, 16), (5, 3)])
def test_verify_tiny(S, T):
    shape = WL.TINY.with_(num_slots=96)
    args = _inputs(shape, S, T, 10000 + 10 * S + T)
    _compare(shape, *args, *_run_verify(shape, *args))


def test_verify_shard_four_tokens():
    shape = WL.SHARD
    args = _inputs(shape, 4, 4, 10100)
    _compare(shape, *args, *_run_verify(shape, *args))


def test_verify_bf16_state_first_layer_with_a_padding_sequence():
    shape = WL.SHARD_BF16
    args = _inputs(shape, 5, 3, 10200, first_layer=True, pad=(2,))
    _compare(shape, *args, *_run_verify(shape, *args))


def test_verify_row_tiles():
    """More rows than one launch takes: whole sequences per launch."""
    shape = WL.TINY.with_(num_slots=96, max_rows=64)
    args = _inputs(shape, 3, 8, 10300)
    _compare(shape, *args, *_run_verify(shape, *args))


def test_verify_equals_successive_decode_steps_bit_for_bit():
    """The verify step's rows and per-token slots equal T decode steps run
    one after another on the GPU, each reading the state the previous one
    stored (rows are batch-invariant, so the projections agree bit for bit)."""
    shape = WL.SHARD
    S, T = 3, 4
    w, st, stp, sin, sout = _inputs(shape, S, T, 10400)
    core, res, conv, ssm = _run_verify(shape, w, st, stp, sin, sout)
    dw = {k: (v.cuda() if v is not None else None) for k, v in w.items()}
    layer = GdnDecode(shape)
    for s in range(S):
        dconv, dssm = st["conv_state"].cuda(), st["ssm_state"].cuda()
        for t in range(T):
            row = s * T + t
            idx = torch.tensor([sin[s]], dtype=torch.int32, device="cuda")
            c1, r1 = layer.step(stp["x"][row:row + 1].cuda(), stp["residual"][row:row + 1].cuda(), dw, idx,
                                dconv, dssm)
            torch.cuda.synchronize()
            assert torch.equal(c1[0].view(torch.int16), core[row].view(torch.int16))
            assert torch.equal(r1[0].view(torch.int16), res[row].view(torch.int16))
            assert torch.equal(dssm[sin[s]].view(torch.int32), ssm[sout[s, t]].view(torch.int32))
            assert torch.equal(dconv[sin[s]].view(torch.int16), conv[sout[s, t]].view(torch.int16))
    assert layer.check()[0] == 0


def test_verify_needs_bf16_weights_on_the_tensor_core_engine():
    from gated_deltanet_layer_gb300 import GdnError, _native
    shape = WL.DENSE_MXFP4
    layer = GdnDecode(shape)
    args = _inputs(shape, 1, 2, 10500)
    w, st, stp, sin, sout = args
    with pytest.raises(GdnError) as e:
        _run_verify(shape, w, st, stp, sin, sout)
    assert e.value.code == _native.GDN_ERR_UNSUPPORTED
