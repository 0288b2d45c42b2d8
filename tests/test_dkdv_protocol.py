"""The barrier protocol of the dK/dV kernel, on a model of its roles
(tests/dkdv_protocol.py): every parity wait within one phase of its barrier
and no shared buffer read early or overwritten while in use, under random
interleavings of the roles, the two tensor-core queues and the asynchronous
copies (uniform, and with a role starved just as its wait is about to
pass), for resident and one-unit CTAs at D = 64 and D = 128, with atomic
and deterministic dQ.  A second test leaves out one wait at a time and checks
that the model then fails: each wait is needed, and the checks catch its
absence."""
import pytest

from dkdv_protocol import CONFIGS, UNIT_PATTERNS, ProtocolError, run_case

SEEDS = 6


@pytest.mark.parametrize("slow", [(), "blocked"])
@pytest.mark.parametrize("independent_signal", [False, True])
def test_protocol_holds_under_random_interleavings(independent_signal, slow):
    runs = 0
    for units in UNIT_PATTERNS:
        for config in CONFIGS:
            for seed in range(SEEDS):
                run_case(units, config, seed, independent_signal=independent_signal, slow=slow)
                runs += 1
    assert runs == len(UNIT_PATTERNS) * len(CONFIGS) * SEEDS


# The waits of the protocol, by role.  Not listed: the elementwise warps'
# wait for their tile's Q / dO stage, which the model shows is implied by the
# S^T products having read that stage, but which in the kernel is also what
# makes the stage's LSE / Di rows (written by the copy engine) visible to
# those warps' own loads, an ordering the model does not represent; the
# resident epilogue's waits for the last two dQ^T products before it stages
# dK, dV over their dS^T tiles, implied by its wait for the accumulators (the
# gradient warp commits that barrier after issuing those products, and a
# commit completes only when all of the thread's earlier products have;
# kept in the kernel as a cheap guard); the score warp's wait, at a resident
# CTA's unit boundary, for the previous unit's last dV, dK to be issued, which
# orders the tensor-core queue for speed only; and the bulk-reduction issuer's wait
# for its staging warps and the final drains, without which the model
# deadlocks or reads a stage never written.
WAITS = [
    "prod.kv_empty", "prod.qdo_empty", "prod.buf_ready",
    "score.kv_full", "score.buf_ready",
    "grad.s_read", "grad.p_full", "grad.ds_last",
    "buf.dq_full", "buf.qdo_full", "buf.buf_ready", "buf.stage_free",
    "elem.s_full", "elem.dq_full", "elem.epi_read",
    "epi.acc_full", "epi.epi_read",
]


@pytest.mark.parametrize("wait", WAITS)
def test_each_wait_is_needed(wait):
    # The waits on epi_read guard the seven warps that do not signal it; the
    # model's elementwise role includes the signalling thread, so they are
    # checked with the signal as an independent role.
    independent = wait.endswith("epi_read")
    for seed in range(40):
        for slow in ((), "blocked"):
            for units in UNIT_PATTERNS:
                for config in CONFIGS:
                    try:
                        run_case(units, config, seed, skip={wait}, independent_signal=independent,
                                 slow=slow)
                    except ProtocolError:
                        return
    pytest.fail(f"the model passes without {wait}")
