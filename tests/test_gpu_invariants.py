"""GPU invariants the method's own kernel checks name (sgl-amd-mono #89,
"Kernel checks" table): bf16 state against the f32 kernel on the widened
state, batch invariance, graph replay against eager runs, a wait that runs
out setting the deadline error word; plus index errors and the host-side
argument checks of the C ABI."""
import time

import numpy as np
import pytest
import torch

from gated_deltanet_layer_gb300 import GdnDecode, GdnError, _native, workloads as WL
from gdn_harness import Case, compare, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _bits(t):
    return t.contiguous().view(torch.int16).cpu() if t.dtype == torch.bfloat16 else t.contiguous().view(torch.int32).cpu()


@pytest.mark.parametrize("rows", [1, 8])
def test_bf16_state_matches_f32_kernel_on_widened_state(rows):
    """Core and conv state bit-equal to the f32-state launch on the widened
    state; the new bf16 state is the f32 result rounded to bf16."""
    sh16 = WL.SHARD_BF16
    sh32 = WL.SHARD
    case16 = Case(sh16, rows, 6000 + rows, pad_rows=1 if rows > 1 else 0).to_device()
    case32 = Case(sh32, rows, 0, weights=case16.w, state={
        "conv_state": case16.st["conv_state"], "ssm_state": case16.st["ssm_state"].float()},
        step=case16.step).to_device()
    c16, r16 = case16.run_gpu(GdnDecode(sh16))
    c32, r32 = case32.run_gpu(GdnDecode(sh32))
    assert torch.equal(_bits(c16), _bits(c32))
    assert torch.equal(_bits(r16), _bits(r32))
    assert torch.equal(_bits(case16.dconv), _bits(case32.dconv))
    assert torch.equal(_bits(case16.dssm), _bits(case32.dssm.to(torch.bfloat16)))


@pytest.mark.parametrize("shape", [WL.SHARD, WL.FULL], ids=["shard", "full"])
def test_batch_invariance(shape):
    """A probe row's outputs (core, residual_out, its state slot) do not change
    with the other rows, its position or the width. On the full layer the
    wider steps give a CTA several (row, value head) tasks, so the pipelined
    recurrence and the one-task path must agree bit for bit."""
    base = Case(shape, 16, 6100)
    probe_x = base.step["x"][0].clone()
    probe_r = base.step["residual"][0].clone()
    probe_slot = int(base.step["state_indices"][0])
    outs = []
    for width, pos, seed in [(1, 0, 1), (3, 2, 2), (8, 5, 3), (16, 15, 4), (16, 0, 5), (9, 4, 6)]:
        stp = WL.make_step(shape, width, 6200 + seed)
        stp["x"][pos] = probe_x
        stp["residual"][pos] = probe_r
        idx = stp["state_indices"]
        idx[idx == probe_slot] = 0  # keep slots distinct
        idx[pos] = probe_slot
        case = Case(shape, width, 0, weights=base.w, state=base.st, step=stp).to_device()
        core, res = case.run_gpu(GdnDecode(shape))
        outs.append((_bits(core[pos]), _bits(res[pos]), _bits(case.dssm[probe_slot]),
                     _bits(case.dconv[probe_slot])))
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert torch.equal(a, b)


def test_graph_replay_matches_eager():
    """Widths 8, 1, 3, 8, 2, 5 captured in one CUDA graph on one state, replayed
    200 times (the replay count of sgl-amd-mono #89, Kernel checks); every
    output and the final states bit-equal to the same sequence run eagerly
    200 times."""
    shape = WL.SHARD
    widths = [8, 1, 3, 8, 2, 5]
    base = Case(shape, 8, 6300)
    steps = [WL.make_step(shape, w, 6400 + i) for i, w in enumerate(widths)]
    dw = {k: (v.cuda() if v is not None else None) for k, v in base.w.items()}
    xs = [(s["x"].cuda(), s["residual"].cuda(), s["state_indices"].cuda()) for s in steps]
    reps = 200

    def run(graph):
        conv = base.st["conv_state"].cuda()
        ssm = base.st["ssm_state"].cuda()
        layer = GdnDecode(shape)
        outs = [(torch.empty(w, shape.num_v_heads * shape.head_v_dim, dtype=torch.bfloat16, device="cuda"),
                 torch.empty(w, shape.hidden, dtype=torch.bfloat16, device="cuda")) for w in widths]
        ws = layer.weights_struct(dw)

        def seq():
            for (x, r, i), (c, ro) in zip(xs, outs):
                layer.step(x, r, dw, i, conv, ssm, c, ro, weights_struct=ws)

        if graph:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(s):
                with torch.cuda.graph(g, stream=s):
                    seq()
            torch.cuda.current_stream().wait_stream(s)
            for _ in range(reps):
                g.replay()
        else:
            for _ in range(reps):
                seq()
        torch.cuda.synchronize()
        assert layer.check()[0] == 0
        return conv, ssm, outs

    ce, se, oe = run(False)
    cg, sg, og = run(True)
    assert torch.equal(_bits(ce), _bits(cg))
    assert torch.equal(_bits(se), _bits(sg))
    for (a, b), (c, d) in zip(oe, og):
        assert torch.equal(_bits(a), _bits(c)) and torch.equal(_bits(b), _bits(d))


def test_stalled_wait_sets_deadline_word_and_returns():
    """CTA 0 never publishes its norm partials: every CTA's first wait gives up
    at the deadline, the error word names the norm wait, the launch returns,
    and later launches return at once without touching state until reset."""
    shape = WL.SHARD
    case = Case(shape, 4, 6500).to_device()
    layer = GdnDecode(shape, deadline_us=20000, debug_flags=_native.GDN_DEBUG_SKIP_NORM_PUBLISH)
    ssm0 = case.dssm.clone()
    conv0 = case.dconv.clone()
    torch.cuda.synchronize()
    t0 = time.time()
    case.run_gpu(layer)
    st, detail = layer.check()
    elapsed = time.time() - t0
    assert st == _native.GDN_ERR_DEADLINE
    assert (detail >> 16) & 0xff == 1  # the norm wait
    assert elapsed < 5.0
    assert torch.equal(case.dssm, ssm0) and torch.equal(case.dconv, conv0)
    # sticky: the next launch returns at once and writes nothing
    core = torch.full((4, shape.num_v_heads * shape.head_v_dim), 7.0, dtype=torch.bfloat16, device="cuda")
    layer.step(case.dx, case.dres, case.dw, case.didx, case.dconv, case.dssm, core_out=core)
    assert layer.check()[0] == _native.GDN_ERR_DEADLINE
    assert torch.all(core == 7.0)
    layer.reset()
    assert layer.check() == (0, 0)
    # a healthy handle on the same tensors still matches the oracle
    good = GdnDecode(shape)
    c, r = case.run_gpu(good)
    assert good.check()[0] == 0
    compare(case, case.run_oracle(), c, r)


def test_index_out_of_range_sets_index_error_and_pads_the_row():
    shape = WL.TINY.with_(num_slots=32)
    case = Case(shape, 5, 6600)
    case.step["state_indices"][2] = shape.num_slots
    case.to_device()
    layer = GdnDecode(shape)
    core, res = case.run_gpu(layer)
    st, detail = layer.check()
    assert st == _native.GDN_ERR_INDEX and (detail & 0xffff) == 2
    compare(case, case.run_oracle(), core, res)


def test_host_argument_errors():
    shape = WL.TINY.with_(num_slots=32, max_rows=4)
    case = Case(shape, 4, 6700).to_device()
    layer = GdnDecode(shape)
    with pytest.raises(GdnError):  # rows beyond max_rows
        big = torch.zeros(5, shape.hidden, dtype=torch.bfloat16, device="cuda")
        layer.step(big, big.clone(), case.dw, torch.arange(1, 6, dtype=torch.int32, device="cuda"),
                   case.dconv, case.dssm)
    buf = torch.zeros(4 * shape.hidden + 8, dtype=torch.bfloat16, device="cuda")
    mis = buf[1:1 + 4 * shape.hidden].view(4, shape.hidden)  # 2-byte offset
    with pytest.raises(GdnError):
        layer.step(mis, case.dres, case.dw, case.didx, case.dconv, case.dssm)
    with pytest.raises(GdnError):  # residual_out aliases x
        layer.step(case.dx, case.dres, case.dw, case.didx, case.dconv, case.dssm, residual_out=case.dx)
    with pytest.raises(GdnError):  # core_out inside the ssm state
        layer.step(case.dx, case.dres, case.dw, case.didx, case.dconv, case.dssm,
                   core_out=case.dssm.view(torch.bfloat16).view(-1)[:4 * 512].view(4, 512))
    assert layer.check()[0] == 0  # nothing was launched


def test_no_early_weights_sees_weights_written_by_the_kernel_just_before():
    """With GDN_LAUNCH_NO_EARLY_WEIGHTS the step reads nothing before the
    kernel launched just before it in the stream has finished. Torch kernels
    (dtype-converting copies, so they run as kernels rather than copy-engine
    transfers) overwrite in_proj_qkvz, in_proj_ba and the input-norm weight
    right before each step; every step matches the oracle on the new weights."""
    shape = WL.SHARD
    case = Case(shape, 4, 6800).to_device()
    layer = GdnDecode(shape, launch_flags=_native.GDN_LAUNCH_NO_EARLY_WEIGHTS)
    fresh = WL.make_weights(shape, 6801)
    src = {k: fresh[k].float().cuda() for k in ("qkvz", "ba", "input_norm_w")}
    # a first step on the old weights (tile maps encoded, module warm)
    case.run_gpu(layer)
    conv0, ssm0 = case.st["conv_state"].cuda(), case.st["ssm_state"].cuda()
    case.dconv.copy_(conv0)
    case.dssm.copy_(ssm0)
    torch.cuda.synchronize()
    for k, t in src.items():
        case.dw[k].copy_(t)  # f32 -> bf16: a kernel, launched just before the step
    core, res = layer.step(case.dx, case.dres, case.dw, case.didx, case.dconv, case.dssm)
    torch.cuda.synchronize()
    assert layer.check()[0] == 0
    for k in src:
        case.w[k] = fresh[k]
    compare(case, case.run_oracle(), core, res)
