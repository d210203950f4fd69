"""The fp64 oracle against results fixed by mathematics (CPU only)."""
import numpy as np
import pytest

import oracle
from tests import oracle_pins as pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.ssd_recurrence)


def test_chunk_cumsum_entries():
    """oracle.chunk_cumsum, every interior entry, against products of the
    per-step decay factors (pin p11)."""
    pins.pin_chunk_cumsum(oracle.chunk_cumsum)


def _cumsum_layout(dt, A, Q, order):
    dt = np.asarray(dt, np.float64)
    b, L, H = dt.shape
    dA = (dt * A[None, None, :]).reshape(b, L // Q, Q, H)
    return order(dA).transpose(0, 3, 1, 2).copy()


CUMSUM_MUTANTS = {
    # reversed inside the chunk: the chunk totals (last entries) are unchanged
    "reversed_in_chunk": lambda dt, A, Q: _cumsum_layout(
        dt, A, Q, lambda d: np.cumsum(d[:, :, ::-1, :], axis=2)),
    # exclusive running sum
    "exclusive": lambda dt, A, Q: _cumsum_layout(
        dt, A, Q, lambda d: np.cumsum(d, axis=2) - d),
    # steps and heads strided the wrong way round inside a chunk
    "head_shifted": lambda dt, A, Q: _cumsum_layout(
        dt, np.roll(A, 1), Q, lambda d: np.cumsum(d, axis=2)),
    # one step late: the decay of step q taken from step q - 1
    "step_shifted": lambda dt, A, Q: _cumsum_layout(
        np.roll(dt, 1, axis=1), A, Q, lambda d: np.cumsum(d, axis=2)),
}


@pytest.mark.parametrize("name", sorted(CUMSUM_MUTANTS))
def test_cumsum_pin_catches_mutant(name):
    with pytest.raises(AssertionError):
        pins.pin_chunk_cumsum(CUMSUM_MUTANTS[name])


@pytest.mark.parametrize("L,Q", [(64, 1), (64, 4), (64, 16), (64, 32), (60, 16), (61, 25)])
def test_stage_definitions_match_chunked_algorithm(L, Q):
    """The per-stage oracle intermediates (cumulative decay, chunk-local
    states, states entering each chunk) equal the stage values of the chunked
    algorithm written out independently in oracle_pins.chunked_form, a
    partial last chunk included (its missing cumsum entries repeat the last
    one: dt = 0 steps)."""
    x, dt, A, B, C, D, s0 = pins.small_problem(21, b=2, L=L, H=4, P=3, N=5, G=2)
    _, fin, cums, locs, ins = pins.chunked_form(x, dt, A, B, C, D, s0, Q)
    nc = -(-L // Q)
    cum = oracle.chunk_cumsum(dt, A, Q)
    st = oracle.chunk_states(x, dt, A, B, Q)
    sin, f2 = oracle.states_entering(x, dt, A, B, C, Q, s0)
    assert cum.shape == (2, 4, nc, Q) and st.shape == (2, nc, 4, 3, 5) and sin.shape == st.shape
    for b in range(2):
        for h in range(4):
            for c in range(nc):
                n = len(cums[b, h, c])
                pins._close(cum[b, h, c, :n], cums[b, h, c], what="cumsum")
                assert np.all(cum[b, h, c, n:] == cum[b, h, c, n - 1])
                pins._close(st[b, c, h], locs[b, h, c], what="chunk state")
                pins._close(sin[b, c, h], ins[b, h, c], what="state entering chunk")
    pins._close(f2, fin, what="final")


def test_snapshots_of_zero_input_are_pure_decay():
    """With x = 0 the state entering chunk c is exp(sum of all earlier dt*A)
    times the initial state: ties the cumulative decay to the recurrence."""
    x, dt, A, B, C, D, s0 = pins.small_problem(22, b=1, L=48, H=2, P=2, N=3, G=1)
    sin, _ = oracle.states_entering(np.zeros_like(x), dt, A, B, C, 16, s0)
    cum = oracle.chunk_cumsum(dt, A, 16)                 # [1, H, 3, 16]
    total = np.concatenate([np.zeros((1, 2, 1)), np.cumsum(cum[:, :, :, -1], axis=2)[:, :, :-1]], axis=2)
    for c in range(3):
        want = np.exp(total[0, :, c])[:, None, None] * s0[0]
        pins._close(sin[0, c], want, what=f"pure decay chunk {c}")


def test_empty_sequence():
    x = np.zeros((1, 0, 2, 3))
    y, f = oracle.ssd_recurrence(x, np.zeros((1, 0, 2)), -np.ones(2), np.zeros((1, 0, 1, 4)),
                                 np.zeros((1, 0, 1, 4)), np.ones(2), np.ones((1, 2, 3, 4)))
    assert y.shape == (1, 0, 2, 3)
    assert np.array_equal(f, np.ones((1, 2, 3, 4)))


def test_rejects_bad_groups():
    with pytest.raises(ValueError):
        oracle.ssd_recurrence(np.zeros((1, 4, 3, 2)), np.zeros((1, 4, 3)), -np.ones(3),
                              np.zeros((1, 4, 2, 2)), np.zeros((1, 4, 2, 2)))
