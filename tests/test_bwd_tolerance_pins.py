"""The backward tolerance of dweight/dbias on the five workloads, pinned.

Its FP32 term is gamma * S with gamma = (D + 64) 2^-24, where D is the
longest addition chain of a parameter-gradient term in the kernel that runs
(oracle/compare.py, ``reduction_depth``), which follows from the backward
partition plan.  The plan is a host-side function of the layout class and the
sizes (the workspace size the library reports encodes it), so these tests run
without a GPU.  Pinning D for each workload means that a plan change which
lengthens the chains fails here instead of loosening the bar unnoticed; and
every workload's gamma stays below 2^-15.
"""
import pytest

from causal_depthwise_conv1d_gb300 import inputs
from oracle import compare

# workload: B, C, L, K, dtype, x strides (elements), then the pinned plan:
# gradient kernel, partials P = B * partitions, chain length D
WORKLOADS = {
    1: (1, 64, 512, 4, "f32", (32768, 512, 1), "bwd_time", 1, 24),
    2: (8, 5120, 2048, 4, "bf16", (10485760, 2048, 1), "bwd_time", 8, 47),
    3: (4, 5120, 4096, 4, "bf16", (41943040, 1, 10240), "bwd_chlast", 60, 307),
    4: (1, 4096, 16384, 4, "f16", (67108864, 1, 4096), "bwd_chlast", 74, 242),
    5: (1, 16, 4194304, 3, "f32", (67108864, 4194304, 1), "bwd_time", 2048, 134),
}
DT = {"f32": 0, "f16": 1, "bf16": 2}


@pytest.fixture(scope="module")
def ccv():
    from causal_depthwise_conv1d_gb300 import build
    build.build()
    import causal_depthwise_conv1d_gb300 as ccv
    ccv.load_library()
    return ccv


@pytest.mark.parametrize("cfg", sorted(WORKLOADS))
def test_reduction_depth_of_each_workload_is_pinned(ccv, cfg):
    B, C, L, K, dtype, xs, want_kernel, want_P, want_D = WORKLOADS[cfg]
    # dout and dx dense in x's fast dimension, as the tests and the bench make them
    if xs[2] == 1:
        ds, kernel = (C * L, L, 1), "bwd_time"
    else:
        ds, kernel = (L * C, 1, C), "bwd_chlast"
    nbytes = ccv.ccv_bwd_workspace_size(xs, ds, ds, B, C, L, K, DT[dtype])
    P = nbytes // ((K + 1) * C * 4)
    assert (kernel, P) == (want_kernel, want_P)
    assert compare.reduction_depth(kernel, B, L, P) == want_D
    assert compare.gamma_dw(kernel, B, L, P) < 2.0 ** -15


def test_the_table_matches_the_workload_definitions():
    """The shapes above are the seeded workloads': sizes and dtype against the
    workload names, and the strides of the small one, whose data is cheap to
    make."""
    import re
    for i, name in enumerate(inputs.CONFIG_NAMES, start=1):
        m = re.match(r"c\d_(\w+?)_.*_B(\d+)_C(\d+)_L(\d+)_K(\d)", name)
        dt, B, C, L, K = m.group(1), *(int(m.group(j)) for j in range(2, 6))
        assert (B, C, L, K, dt) == WORKLOADS[i][:5], name
    p = inputs.make_config(1)
    xv = p.x_view()
    assert (p.B, p.C, p.L, p.K, p.dtype) == WORKLOADS[1][:5]
    assert tuple(s // xv.itemsize for s in xv.strides) == WORKLOADS[1][5]
