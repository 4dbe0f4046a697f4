"""gdn_decode_step_static against gdn_decode_step on the same inputs, through
the C ABI.

The static entry point is for callers that cannot allocate device memory (a
host program with no device allocator of its own, or a runtime whose memory
all belongs to its own pool): it runs the same kernel on a fixed scratch
array inside the library instead of a caller workspace, with no handle.

Each case runs two steps in a row on each path from the same starting state,
so the second step reads the state the first one wrote and runs on counters
the first one advanced. Both paths launch the same kernel with the same plan
and a fixed reduction order, so every output must be bit-identical; the
first step is also compared with the CPU oracle at the step's tolerances.
This file is named to be collected last: the static scratch lives as long as
the process, and the cases must pass both alone and after every other GPU
test."""
import pytest
import torch

from gated_deltanet_layer_gb300 import GdnDecode, GdnError, _native, step_static, workloads as WL
from gdn_harness import Case, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _bits(t):
    return t.contiguous().view(torch.int16 if t.element_size() == 2 else torch.int32)


def _two_steps_each(shape, rows, seed, **kw):
    case = Case(shape, rows, seed, **kw).to_device()
    nxt = Case(shape, rows, seed + 50, **kw).to_device()
    # the second step uses the same slots, so it reads the state the first wrote
    steps = [(case.dx, case.dres, case.didx), (nxt.dx, nxt.dres, case.didx)]

    layer = GdnDecode(shape)
    conv_a, ssm_a = case.dconv.clone(), case.dssm.clone()
    ref = []
    for k, (x, r, i) in enumerate(steps):
        core, res_out = layer.step(x, r, case.dw, i, conv_a, ssm_a)
        ref.append((core.clone(), res_out.clone()))
        if k == 0:
            # the handle path's first step against the oracle
            torch.cuda.synchronize()
            case.dconv, case.dssm, saved = conv_a.clone(), ssm_a.clone(), (case.dconv, case.dssm)
            compare(case, case.run_oracle(), core, res_out)
            case.dconv, case.dssm = saved
    assert layer.check()[0] == 0

    conv_b, ssm_b = case.dconv.clone(), case.dssm.clone()
    core_b = torch.empty(rows, shape.num_v_heads * shape.head_v_dim, dtype=torch.bfloat16, device="cuda")
    res_b = torch.empty(rows, shape.hidden, dtype=torch.bfloat16, device="cuda")
    ws = GdnDecode.weights_struct(case.dw)
    got = [(torch.empty_like(core_b), torch.empty_like(res_b)) for _ in steps]
    torch.cuda.synchronize()
    reserved0 = torch.cuda.memory_reserved()
    free_before = torch.cuda.mem_get_info()[0]
    for k, (x, r, i) in enumerate(steps):
        if k == 1:
            torch.cuda.synchronize()
            free_second = torch.cuda.mem_get_info()[0]
        st, detail = step_static(shape, x, r, ws, i, conv_b, ssm_b, core_b, res_b, check=True)
        assert st == _native.GDN_OK, f"device error 0x{detail:08x}"
        got[k][0].copy_(core_b)
        got[k][1].copy_(res_b)
    torch.cuda.synchronize()
    # nothing went through torch's allocator on either call
    assert torch.cuda.memory_reserved() == reserved0
    # the second call found its set-up done: no device memory changed hands.
    # The device-wide free count is only a bound (another process could move
    # it): an allocation by the call would take at least one 2 MiB granule.
    # The first call may load the library's module that holds the scratch
    # array (lazy module loading), which the driver does, not the call: a
    # loose bound of the array's size plus a few MiB of code and tables.
    assert abs(torch.cuda.mem_get_info()[0] - free_second) < (2 << 20)
    assert free_before - free_second <= _native.GDN_STATIC_SCRATCH_BYTES + (16 << 20)

    for (ca, ra), (cb, rb) in zip(ref, got):
        assert torch.equal(_bits(ra), _bits(rb))
        assert torch.equal(_bits(ca), _bits(cb))
    assert torch.equal(_bits(ssm_a), _bits(ssm_b))
    assert torch.equal(_bits(conv_a), _bits(conv_b))


@pytest.mark.parametrize("rows", [1, 16])
def test_static_scratch_matches_workspace_path_shard(rows):
    _two_steps_each(WL.SHARD, rows, 7000 + rows)


def test_static_scratch_matches_workspace_path_tiny_first_layer_pad_rows():
    # another config: the set-up runs again on the same scratch
    _two_steps_each(WL.TINY.with_(num_slots=32), 8, 7100, first_layer=True, pad_rows=2)


def test_static_scratch_bf16_state():
    _two_steps_each(WL.SHARD_BF16, 5, 7200)


def test_static_scratch_rejects_a_layer_that_does_not_fit():
    # the full 8192-wide layer: its projection partials alone need ~32 MB.
    # Two state slots keep the buffers of the (never launched) step small
    # but correctly sized.
    shape = WL.FULL.with_(num_slots=2)
    case = Case(shape, 1, 7300).to_device()
    core = torch.empty(1, shape.num_v_heads * shape.head_v_dim, dtype=torch.bfloat16, device="cuda")
    res = torch.empty(1, shape.hidden, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(GdnError) as e:
        step_static(shape, case.dx, case.dres, case.dw, case.didx, case.dconv, case.dssm, core, res)
    assert e.value.code == _native.GDN_ERR_UNSUPPORTED
