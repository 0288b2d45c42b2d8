"""The barrier protocol of the deterministic dQ kernel, on a model of its
roles (tests/dq_protocol.py): every parity wait within one phase and no
buffer read early or overwritten while in use, under random interleavings;
and each wait left out in turn makes the model fail."""
import pytest

from dq_protocol import TILE_COUNTS, DqPipeline, ProtocolError


def test_protocol_holds_under_random_interleavings():
    for n in TILE_COUNTS:
        for seed in range(12):
            DqPipeline(n, seed).run()


# Not listed: the elementwise warps' wait for Q / dO and their LSE / Di rows,
# which the model shows is implied by their wait for the first scores (the
# score products read Q after it landed), but which in the kernel makes the
# copied LSE / Di rows visible to those warps' own loads.
WAITS = ["prod.kv_empty", "relay.kv_full", "score.q_full", "score.buf_ready", "grad.p_full",
         "elem.s_full", "epi.all_done"]


@pytest.mark.parametrize("wait", WAITS)
def test_each_wait_is_needed(wait):
    for seed in range(60):
        for n in TILE_COUNTS:
            try:
                DqPipeline(n, seed, skip={wait}).run()
            except ProtocolError:
                return
    pytest.fail(f"the model passes without {wait}")
