"""The bounded barrier waits of the channel-last TMA kernel, made to run out
without a fault: ccv_test_bounded_wait shortens the wait budget of one launch
and leaves out one tensor copy of its first warp (the copy is never issued, so
nothing is in flight that could fault).  The warp's wait runs out, it records
the consumer-wait bit, waits for the copy it did issue and returns; the next
ordinary call on the same stream is complete and matches the oracle."""
import pytest

from causal_depthwise_conv1d_gb300 import inputs
from tests import parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU-only machines
    pytest.skip("needs a CUDA device", allow_module_level=True)

# consumer wait (1): the warp gave up on the left-out stage; drain wait (4)
# would mean it also gave up on a copy it did issue
CONSUMER_WAIT = 1
BUDGET = 1 << 21  # about 1 ms at the GB300's SM clock; a staged copy lands in microseconds


def _case(seed):
    # 8 bands x 4096 rows: the first warp's share is 5 units = 2 stages, so
    # with stage 0 left out, stage 1 is in flight when the wait runs out
    return inputs.make_case(seed, 1, 2048, 4096, 4, "bf16", activation="silu", layout="channel", final=True)


@pytest.mark.parametrize("skip_stage", [0, 1])
def test_wait_runs_out_and_the_next_call_is_whole(skip_stage):
    import causal_depthwise_conv1d_gb300 as ccv
    from causal_depthwise_conv1d_gb300 import device as dv

    assert ccv.ccv_device_fault() == 0
    p = _case(14000 + skip_stage)
    d = dv.to_device(p)
    ccv.ccv_test_bounded_wait(BUDGET, skip_stage)
    ccv.ccv_fwd(d.x, d.weight, d.bias, None, None, final_states_out=d.final_states, activation="silu", out=d.out)
    assert ccv.ccv_last_kernel() == "chlast_tma"
    torch.cuda.synchronize()
    assert ccv.ccv_device_fault() == CONSUMER_WAIT
    # the setting was one-shot: the same stream's next call is ordinary
    parity.check_problem(p, expect_kernel="chlast_tma")


def test_a_cleared_setting_leaves_the_next_call_alone():
    import causal_depthwise_conv1d_gb300 as ccv

    ccv.ccv_test_bounded_wait(BUDGET, 0)
    ccv.ccv_test_bounded_wait(0, 0)  # clears it
    parity.check_problem(_case(14010), expect_kernel="chlast_tma")
