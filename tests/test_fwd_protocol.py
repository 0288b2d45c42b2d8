"""The barrier protocol of the forward kernel, on a model of its roles
(tests/fwd_protocol.py): every parity wait within one phase of its barrier
and no buffer read early or overwritten while in use, under random
interleavings (uniform, and with a role starved just as its wait is about to
pass), for resident and one-unit CTAs over causal, non-causal,
windowed and ragged bands.  A second test leaves out one wait at a time and
checks that the model then fails."""
import pytest

from fwd_protocol import BANDS, FwdPipeline, ProtocolError, units_for

SEEDS = 4


def cases():
    for n, wl, wr in BANDS:
        for heads in (1, 3):
            units = units_for(n, wl, wr, heads)
            for u in units[:2]:
                yield [u], False
            yield units, True


@pytest.mark.parametrize("slow", [(), "blocked"])
def test_protocol_holds_under_random_interleavings(slow):
    runs = 0
    for units, resident in cases():
        for seed in range(SEEDS):
            FwdPipeline(units, resident, seed, slow=slow).run()
            runs += 1
    assert runs > 100


# Not listed: the wait a softmax group makes before rescaling O for the
# previous tile's P V product, which the model shows is implied by its wait
# for the next scores (S_t(j) is issued after P V_t(j - 1) by the same thread,
# and the commit that completes s_full covers every earlier product of that
# thread); the kernel keeps it as a guard on a rarely taken path.
WAITS = ["prod.q_empty", "prod.k_empty", "prod.v_empty",
         "mma.q_full", "mma.k_full", "mma.v_full", "mma.p_full",
         "sm.s_full", "epi.o_done"]


@pytest.mark.parametrize("wait", WAITS)
def test_each_wait_is_needed(wait):
    for seed in range(30):
        for slow in ((), "blocked"):
            for units, resident in cases():
                try:
                    FwdPipeline(units, resident, seed, skip={wait}, slow=slow).run()
                except ProtocolError:
                    return
    pytest.fail(f"the model passes without {wait}")
