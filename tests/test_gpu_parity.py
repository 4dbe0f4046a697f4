"""CUDA path (through the C ABI) against the CPU oracle, element by element,
on seeded synthetic layers of every workload shape: widths 1..16, pad rows,
the first-layer variant and the bf16 state."""
import numpy as np
import pytest
import torch

from gated_deltanet_layer_gb300 import GdnDecode, workloads as WL
from gdn_harness import Case, compare, f64

pytestmark = pytest.mark.gpu

ENGINES = ["tcgen05", "cuda_core"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _run(shape, rows, seed, engine, **kw):
    case = Case(shape, rows, seed, **kw).to_device()
    layer = GdnDecode(shape, engine=engine)
    core, res_out = case.run_gpu(layer)
    st, detail = layer.check()
    assert st == 0, f"device error 0x{detail:08x}"
    compare(case, case.run_oracle(), core, res_out)


TINY32 = WL.TINY.with_(num_slots=32)


@pytest.mark.parametrize("engine", ENGINES)
@pytest.mark.parametrize("rows", [1, 2, 3, 5, 8, 13, 16])
def test_tiny_layer(rows, engine):
    _run(TINY32, rows, 1000 + rows, engine)


@pytest.mark.parametrize("engine", ENGINES)
@pytest.mark.parametrize("rows", [1, 4, 11, 16])
def test_tiny_layer_pad_rows_and_first_layer(rows, engine):
    _run(TINY32, rows, 1100 + rows, engine, first_layer=True, pad_rows=WL.default_pad_rows(rows))


@pytest.mark.parametrize("engine", ENGINES)
def test_tiny_layer_config_slots(engine):
    # the tiny workload as specified: 16 slots, one row
    _run(WL.TINY, 1, 1200, engine)


@pytest.mark.parametrize("engine", ENGINES)
@pytest.mark.parametrize("rows", [1, 2, 4, 8, 16])
def test_shard_layer(rows, engine):
    _run(WL.SHARD, rows, 2000 + rows, engine)


@pytest.mark.parametrize("engine", ENGINES)
@pytest.mark.parametrize("rows", [1, 3, 8, 9, 16])
def test_shard_bf16_state_first_layer_with_pad_rows(rows, engine):
    _run(WL.SHARD_BF16, rows, 3000 + rows, engine, first_layer=True, pad_rows=WL.default_pad_rows(rows))


@pytest.mark.parametrize("engine", ENGINES)
@pytest.mark.parametrize("rows", [3, 16])
def test_shard_bf16_state_with_residual(rows, engine):
    _run(WL.SHARD_BF16, rows, 3100 + rows, engine)


@pytest.mark.parametrize("engine", ENGINES)
@pytest.mark.parametrize("rows", [1, 16])
def test_full_layer(rows, engine):
    _run(WL.FULL, rows, 4000 + rows, engine)


# Stress case: conv weights ~N(0, 0.5) (25x the recipe's) make the v path and
# the state update matter. A projection output that the kernel's f32 sum
# rounds to the other bf16 neighbour than the oracle's exact sum (one ulp, up
# to 2^-5 for |p| in [4, 8)) then moves v by |w3| * ulp ~ 0.5 * 0.03 and the
# state by |k_i| * beta * that ~ 1.4e-3, past the 1e-3 bar of the recipe's
# inputs. The test shows that this is the only source of the excess: with
# the kernel's own q, k, v projection values (read back from the new conv
# taps, each within one bf16 ulp of the oracle's) fed through the oracle's
# conv, norms, gates and delta rule, the kernel's f32 state is within the
# 1e-3 bar; end to end it is within 5e-3.
STRESS_STATE_TOL = 5e-3


def _state_given_kernel_projections(case, gconv):
    """The oracle's f32 state after the step when its q, k, v projection
    outputs are replaced by the kernel's (the new conv taps hold them as
    bf16), b, a and z staying the oracle's. Also checks that each of the
    kernel's values is within one bf16 ulp of the oracle's."""
    from oracle import gdn_oracle as O
    from gdn_harness import bf16_ulp
    sh = case.shape
    Hk, Hv, dk, dv, C = sh.num_k_heads, sh.num_v_heads, sh.head_k_dim, sh.head_v_dim, sh.conv_channels
    ref = case.run_oracle()
    w = {k: f64(v) for k, v in case.w.items()}
    conv0, ssm0 = f64(case.st["conv_state"]), f64(case.st["ssm_state"])
    out = ssm0.copy()
    _, _, _, _, b, a = O.split_projection(ref["p_qkvz"], ref["p_ba"], Hk, Hv, dk, dv)
    for r, s in enumerate(case.step["state_indices"].numpy()):
        if not 0 < s < sh.num_slots:
            continue
        u = gconv[s][:, -1]
        assert np.all(np.abs(u - ref["p_qkvz"][r, :C]) <= bf16_ulp(ref["p_qkvz"][r, :C]))
        y, _ = O.conv_update(conv0[s], w["conv_w"], u)
        qn = O.l2norm(y[:Hk * dk].reshape(Hk, dk), sh.l2_eps) * sh.scale_q
        kn = O.l2norm(y[Hk * dk:2 * Hk * dk].reshape(Hk, dk), sh.l2_eps)
        yv = y[2 * Hk * dk:].reshape(Hv, dv)
        g, beta = O.gates(a[r], b[r], w["A_log"], w["dt_bias"])
        for h in range(Hv):
            kh = h // (Hv // Hk)
            S, _ = O.delta_rule(ssm0[s, h], kn[kh], yv[h], qn[kh], g[h], beta[h])
            out[s, h] = O.f32_round(S)
    return out


def _run_stress(shape, rows, seed, engine, **kw):
    case = Case(shape, rows, seed, **kw).to_device()
    layer = GdnDecode(shape, engine=engine)
    core, res_out = case.run_gpu(layer)
    assert layer.check()[0] == 0
    compare(case, case.run_oracle(), core, res_out, state_tol=STRESS_STATE_TOL)
    cond = _state_given_kernel_projections(case, f64(case.dconv))
    assert float(np.max(np.abs(f64(case.dssm) - cond))) <= 1e-3


@pytest.mark.parametrize("engine", ENGINES)
@pytest.mark.parametrize("shape", [TINY32, WL.SHARD])
def test_strong_conv_weights_and_unit_q_scale(shape, engine):
    _run_stress(shape.with_(q_scale=1.0), 6, 5000, engine, conv_std=0.5)


@pytest.mark.parametrize("engine", ENGINES)
def test_all_rows_pad(engine):
    shape = TINY32
    case = Case(shape, 4, 5100)
    case.step["state_indices"] = torch.tensor([0, -1, 0, -7], dtype=torch.int32)
    case.to_device()
    layer = GdnDecode(shape, engine=engine)
    core, res_out = case.run_gpu(layer)
    assert layer.check()[0] == 0
    compare(case, case.run_oracle(), core, res_out)


@pytest.mark.parametrize("shape", [WL.TINY, WL.SHARD, WL.FULL])
def test_auto_engine_is_tensor_core(shape):
    from gated_deltanet_layer_gb300 import GDN_ENGINE_TCGEN05
    assert GdnDecode(shape).launch_info(1)[1] == GDN_ENGINE_TCGEN05


@pytest.mark.parametrize("rows", [1, 16])
def test_cooperative_launch_option(rows):
    """The opt-in cooperative launch computes the same step."""
    from gated_deltanet_layer_gb300 import _native
    case = Case(WL.SHARD, rows, 6000 + rows).to_device()
    layer = GdnDecode(WL.SHARD, launch_flags=_native.GDN_LAUNCH_COOPERATIVE)
    core, res_out = case.run_gpu(layer)
    assert layer.check()[0] == 0
    compare(case, case.run_oracle(), core, res_out)


# The dense layer with MXFP4 in_proj_qkvz (activations quantised per block of
# 32, W4A4, in_proj_ba bf16 on the unquantised input).
@pytest.mark.parametrize("rows", [1, 6, 16])
def test_dense_mxfp4_layer(rows):
    _run(WL.DENSE_MXFP4, rows, 8000 + rows, "auto")


def test_dense_mxfp4_first_layer_with_pad_rows():
    _run(WL.DENSE_MXFP4, 9, 8100, "tcgen05", first_layer=True, pad_rows=WL.default_pad_rows(9))


# The dense layer with MXFP6 E2M3 in_proj_qkvz (W6A16: bf16 activations).
@pytest.mark.parametrize("rows", [1, 6, 16])
def test_dense_mxfp6_layer(rows):
    _run(WL.DENSE_MXFP6, rows, 8200 + rows, "auto")


def test_dense_mxfp6_first_layer_bf16_state_with_pad_rows():
    _run(WL.DENSE_MXFP6.with_(ssm_dtype="bf16"), 9, 8300, "tcgen05", first_layer=True,
         pad_rows=WL.default_pad_rows(9))


def test_dense_mxfp6_weights_made_as_the_pages_make_them():
    """bf16 weights ~N(0, 0.02) rounded to E2M3 block by block and packed
    (the review comment's steps 2 and 3, by the oracle's quantiser), then
    the whole step against the oracle on the packed weights."""
    from oracle import gdn_oracle as O
    shape = WL.DENSE_MXFP6
    case = Case(shape, 5, 8400)
    dense = WL.make_weights(shape.with_(qkvz_format="bf16"), 8401)["qkvz"].to(torch.float64).numpy()
    codes, scales = O.mxfp6_quantize_matrix(dense)
    case.w["qkvz"] = torch.from_numpy(O.mxfp6_pack(codes))
    case.w["qkvz_scales"] = torch.from_numpy(scales)
    case.to_device()
    layer = GdnDecode(shape)
    core, res_out = case.run_gpu(layer)
    assert layer.check()[0] == 0
    compare(case, case.run_oracle(), core, res_out)


def test_mxfp4_needs_the_tensor_core_engine():
    from gated_deltanet_layer_gb300 import GdnError, _native
    for shape in (WL.DENSE_MXFP4, WL.DENSE_MXFP6):
        with pytest.raises(GdnError) as e:
            GdnDecode(shape, engine="cuda_core")
        assert e.value.code == _native.GDN_ERR_UNSUPPORTED


# Steps wider than one launch's 16 rows run as one launch per tile of 16
# rows (the pages' row cap per launch); every row is checked against the
# oracle, pad rows included.
WIDE_TINY = WL.TINY.with_(num_slots=80, max_rows=64)


@pytest.mark.parametrize("rows", [17, 32, 40, 64])
def test_wide_steps(rows):
    _run(WIDE_TINY, rows, 9000 + rows, "auto", pad_rows=rows // 5)


def test_wide_step_shard_first_layer_bf16_state():
    _run(WL.SHARD_BF16.with_(max_rows=64), 48, 9100, "auto", first_layer=True, pad_rows=12)


def test_wide_step_rows_match_16_row_steps():
    """Each 16-row tile of a 40-row step is bit-identical to a 16-row (or
    8-row) step of the same rows on the same state."""
    shape = WL.SHARD.with_(max_rows=64)
    wide = Case(shape, 40, 9200).to_device()
    cw, rw = wide.run_gpu(GdnDecode(shape))
    for r0 in (0, 16, 32):
        n = min(16, 40 - r0)
        stp = {"x": wide.step["x"][r0:r0 + n].clone(), "residual": wide.step["residual"][r0:r0 + n].clone(),
               "state_indices": wide.step["state_indices"][r0:r0 + n].clone()}
        part = Case(shape, n, 0, weights=wide.w, state=wide.st, step=stp).to_device()
        cp, rp = part.run_gpu(GdnDecode(shape))
        assert torch.equal(cp.view(torch.int16), cw[r0:r0 + n].view(torch.int16))
        assert torch.equal(rp.view(torch.int16), rw[r0:r0 + n].view(torch.int16))
        for s in stp["state_indices"].tolist():
            assert torch.equal(part.dssm[s].view(torch.int32), wide.dssm[s].view(torch.int32))
            assert torch.equal(part.dconv[s].view(torch.int16), wide.dconv[s].view(torch.int16))
