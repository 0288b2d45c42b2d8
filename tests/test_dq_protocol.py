"""The barrier protocol of the deterministic dQ kernel, on a model of its
roles (tests/dq_protocol.py): every parity wait within one phase and no
buffer read early or overwritten while in use, under random interleavings (uniform, and with a role starved just as its
wait is about to pass);
and each wait left out in turn makes the model fail."""
import pytest

from dq_protocol import TILE_COUNTS, DqPipeline, ProtocolError


@pytest.mark.parametrize("slow", [(), "blocked"])
def test_protocol_holds_under_random_interleavings(slow):
    for n in TILE_COUNTS:
        for seed in range(12):
            DqPipeline(n, seed, slow=slow).run()


# Not listed: the elementwise warps' wait for Q / dO and their LSE / Di rows,
# which the model shows is implied by their wait for the first scores (the
# score products read Q after it landed), but which in the kernel makes the
# copied LSE / Di rows visible to those warps' own loads.
WAITS = ["prod.kv_empty", "relay.kv_full", "score.q_full", "score.buf_ready", "grad.p_full",
         "elem.s_full", "epi.all_done"]


@pytest.mark.parametrize("wait", WAITS)
def test_each_wait_is_needed(wait):
    for seed in range(60):
        for slow in ((), "blocked"):
            for n in TILE_COUNTS:
                try:
                    DqPipeline(n, seed, skip={wait}, slow=slow).run()
                except ProtocolError:
                    return
    pytest.fail(f"the model passes without {wait}")
