"""The step with out_proj folded into the launch, through the C ABI, against
the CPU oracle: core and state as for a plain step, and out = bf16(W_o core)."""
import numpy as np
import pytest
import torch

from gated_deltanet_layer_gb300 import GdnDecode, workloads as WL
from gdn_harness import CORE_COS, CORE_MAX_ABS, Case, compare, cosine, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _run(shape, rows, seed, **kw):
    case = Case(shape, rows, seed, **kw)
    case.w["out_proj"] = WL.make_out_proj(shape, seed + 7)
    case.to_device()
    layer = GdnDecode(shape)
    core, res, out = layer.step_out(case.dx, case.dres, case.dw, case.didx, case.dconv, case.dssm)
    torch.cuda.synchronize()
    assert layer.check()[0] == 0
    ref = case.run_oracle()
    compare(case, ref, core, res)
    got, want = f64(out), ref["out"]
    live = [r for r, s in enumerate(case.step["state_indices"].tolist()) if 0 < s < shape.num_slots]
    for r in range(rows):
        if r not in live:
            assert np.all(got[r] == 0.0)
    if live:
        assert cosine(got[live], want[live]) >= CORE_COS
        assert float(np.max(np.abs(got[live] - want[live]))) <= CORE_MAX_ABS
    return case, core, out


@pytest.mark.parametrize("rows", [1, 4, 16])
def test_out_proj_shard(rows):
    _run(WL.SHARD, rows, 11000 + rows)


def test_out_proj_tiny_first_layer_pad_rows():
    _run(WL.TINY.with_(num_slots=32), 7, 11100, first_layer=True, pad_rows=2)


def test_out_proj_full_layer():
    _run(WL.FULL, 2, 11200)


def test_out_proj_dense_mxfp4():
    _run(WL.DENSE_MXFP4, 3, 11300)


def test_out_proj_row_tiles():
    _run(WL.SHARD.with_(max_rows=64), 24, 11400)


def test_out_proj_leaves_core_as_the_plain_step():
    """core_out and the states of the step with out_proj are bit-identical to
    the plain step's on the same inputs."""
    shape = WL.SHARD
    case, core, _ = _run(shape, 6, 11500)
    plain = Case(shape, 6, 11500).to_device()
    c2, _ = plain.run_gpu(GdnDecode(shape))
    assert torch.equal(core.view(torch.int16), c2.view(torch.int16))
    assert torch.equal(case.dssm.view(torch.int32), plain.dssm.view(torch.int32))
