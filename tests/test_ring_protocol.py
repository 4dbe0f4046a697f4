"""A model of the tensor-core engine's weight-ring hand-off with coded
(MXFP4 / MXFP6) weights, run on the CPU over the units of the real plans.

mbarrier waits test a phase parity, so a waiter that is two phases behind a
barrier takes the wrong phase for its own. The model plays the roles of the
kernel against each other in random order with random copy and MMA latencies:
the TMA producer (code tiles into the code ring), eight decode warps (each on
its own: code tile in, bf16 stage released, decode, then one arrival on the
code stage's release and on the stage's `dfull`; at an in_proj_ba unit past
a stage's first use they meet at a barrier and decode warp 0 issues the bf16
tile), and the MMA issuer (waits on `full` or `dfull` of each unit's stage,
each barrier at every one of its phases in order). Every wait that passes is
checked against the phase it is meant for, and the run must end.

The same model of the earlier protocol (the producer issuing the in_proj_ba
tiles and waiting for their stage's release, the decode waiting only for
coded units) shows the aliased waits: the model can find the fault it is
there to exclude."""
import random

import pytest

from gated_deltanet_layer_gb300 import _native, make_config, workloads as WL


class Bar:
    """An mbarrier: `c` completed phases, an arrival count and pending bytes."""

    def __init__(self, count):
        self.c, self.count, self.arr, self.tx = 0, count, 0, 0

    def ok(self, parity):  # try_wait.parity: the phase with this parity has completed
        return (self.c & 1) != parity

    def arrive(self, n=1, tx=0):
        self.arr += n
        self.tx += tx
        self._check()

    def land(self, tx):
        self.tx -= tx
        self._check()

    def _check(self):
        if self.arr == self.count and self.tx == 0:
            self.c, self.arr = self.c + 1, 0


def prefill_units(units, S, R, cap=10):
    coded = n = 0
    while n < min(len(units), cap):
        if units[n]:
            if coded == R:
                break
            coded += 1
        elif n >= S:
            break
        n += 1
    return n


def simulate(units, S, R, seed, current=True, NW=8):
    """Returns the list of protocol errors of one randomised run."""
    rnd = random.Random(seed)
    N = len(units)
    full = [Bar(1) for _ in range(S)]
    dfull = [Bar(NW if current else 1) for _ in range(S)]
    empty = [Bar(1) for _ in range(S)]
    rfull = [Bar(1) for _ in range(R)]
    rempty = [Bar(NW if current else 1) for _ in range(R)]
    kidx, uses_u, uses_c = [], [], []
    k, cu, cc = 0, [0] * S, [0] * S
    for n in range(N):
        kidx.append(k)
        uses_u.append(cu[n % S])
        uses_c.append(cc[n % S])
        if units[n]:
            k += 1
            cc[n % S] += 1
        else:
            cu[n % S] += 1
    events, errors = [], []

    def later(now, fn, span=4.0):
        events.append((now + rnd.random() * span, fn))

    def fill_bf16(now, n):
        full[n % S].arrive(1, tx=1)
        later(now, lambda: full[n % S].land(1))

    def fill_code(now, n):
        r = kidx[n] % R
        rfull[r].arrive(1, tx=1)
        later(now, lambda: rfull[r].land(1))

    pf = prefill_units(units, S, R)
    for n in range(pf):
        (fill_code if units[n] else fill_bf16)(0.0, n)
    prod, mma = pf, 0
    dec = [0] * NW
    passed = [False] * NW
    at_bar = {}

    def step_prod(now):
        nonlocal prod
        if prod >= N:
            return False
        n = prod
        r, rph = kidx[n] % R, (kidx[n] // R) & 1
        if units[n]:
            if not rempty[r].ok(rph ^ 1):
                return False
            if rempty[r].c < kidx[n] // R:
                errors.append(("producer: code stage release aliased", n))
            fill_code(now, n)
        elif not current:
            s, ph = n % S, (n // S) & 1
            if not empty[s].ok(ph ^ 1):
                return False
            if empty[s].c < n // S:
                errors.append(("producer: stage release aliased", n))
            fill_bf16(now, n)
        prod += 1
        return True

    def step_dec(now, w):
        n = dec[w]
        if n >= N:
            return False
        s, ph = n % S, (n // S) & 1
        r, rph = kidx[n] % R, (kidx[n] // R) & 1
        if not units[n]:
            if current and n >= S:
                if not passed[w]:
                    if not empty[s].ok(ph ^ 1):
                        return False
                    if empty[s].c < n // S:
                        errors.append(("decode: stage release aliased", n, w))
                    passed[w] = True
                    at_bar[n] = at_bar.get(n, 0) + 1
                if at_bar[n] < NW:
                    return False
                passed[w] = False
                if w == 0:
                    fill_bf16(now, n)
            elif current and w == 0 and n >= pf:
                fill_bf16(now, n)
            dec[w] += 1
            return True
        if not current and w > 0:  # the earlier protocol: one decoding group
            dec[w] += 1
            return True
        if not (rfull[r].ok(rph) and empty[s].ok(ph ^ 1)):
            return False
        if rfull[r].c < kidx[n] // R + 1:
            errors.append(("decode: code tile aliased", n, w))
        if empty[s].c < n // S:
            errors.append(("decode: stage release aliased", n, w))
        rempty[r].arrive()
        (dfull if current else full)[s].arrive()
        dec[w] += 1
        return True

    def step_mma(now):
        nonlocal mma
        if mma >= N:
            return False
        n = mma
        s = n % S
        if current and units[n]:
            b, want = dfull[s], uses_c[n] + 1
        elif current:
            b, want = full[s], uses_u[n] + 1
        else:
            b, want = full[s], n // S + 1
        if not b.ok((want - 1) & 1):
            return False
        if b.c != want:
            errors.append(("MMA: stage fill aliased", n))
        later(now, lambda: empty[s].arrive(), span=6.0)
        mma += 1
        return True

    now = 0.0
    for _ in range(200000):
        moved = False
        actors = ["p", "m"] + list(range(NW))
        rnd.shuffle(actors)
        for a in actors:
            if rnd.random() < 0.5:
                r = step_prod(now) if a == "p" else step_mma(now) if a == "m" else step_dec(now, a)
                moved = moved or r
        if moved:
            continue
        if not events:
            if mma >= N and prod >= N and min(dec) >= N:
                break
            if not (step_prod(now) or step_mma(now) or any(step_dec(now, w) for w in range(NW))):
                errors.append(("deadlock", prod, mma, tuple(dec)))
                break
            continue
        events.sort(key=lambda e: e[0])
        t, fn = events.pop(0)
        now = max(now, t)
        fn()
    return errors


def _units_of(shape, cta, G=152):
    P = _native.plan(make_config(shape), G)
    ub, nt, KB = P["unit_begin"], P["num_tiles"], P["kblock"]
    tq = shape.n_qkvz // 256
    return [((u // KB) % nt) < tq for u in range(ub[cta], ub[cta + 1])]


def _mixed_ctas(shape, n=12):
    """CTAs whose units mix in_proj_ba (bf16) units with coded ones: where the
    two ways of filling a stage meet."""
    ctas = [c for c in range(152) if len(set(_units_of(shape, c))) == 2]
    assert ctas
    return ctas[:: max(1, len(ctas) // n)]


@pytest.mark.parametrize("shape", [WL.DENSE_MXFP4, WL.DENSE_MXFP6], ids=["mxfp4", "mxfp6"])
@pytest.mark.parametrize("stages", [2, 3])
def test_current_protocol_never_aliases_nor_stalls(shape, stages):
    for cta in _mixed_ctas(shape) + [0, 151]:
        units = _units_of(shape, cta)
        for seed in range(4):
            assert simulate(units, stages, 4, seed * 7919 + cta) == []


def test_the_earlier_protocol_aliases():
    found = []
    for cta in _mixed_ctas(WL.DENSE_MXFP4):
        units = _units_of(WL.DENSE_MXFP4, cta)
        for seed in range(3):
            found += simulate(units, 2, 4, seed * 7919 + cta, current=False)
    assert any("aliased" in e[0] for e in found)
