"""Which kernel layout each width gets (the planner, read through the
testing hook ln_testing_plan): the layouts the measurements chose, and the
invariants every plan must keep (whole warps, the row covered, CTA sizes
within the fitted range), over every 16-byte-aligned width."""

import pytest
import torch

import normalization_fwd_gb300 as nf

pytestmark = pytest.mark.gpu

BF16 = torch.bfloat16


def plan(direction, hidden, dtype=BF16, mode="layernorm", option=False, rows=65536):
    return nf.ln_testing_plan(direction, rows, hidden, dtype, mode, option)


# (direction, hidden, mode, option) -> expected (kind, group, n, block)
EXPECTED = [
    (("forward", 384, "layernorm", True), (4, 16, 3, 256)),     # the bench step's forward
    (("forward", 256, "layernorm", True), (4, 8, 4, 256)),
    (("forward", 512, "rmsnorm", True), (4, 16, 4, 256)),
    (("forward", 1536, "layernorm", True), (5, 64, 3, 64)),     # row-fitted CTAs
    (("forward", 2560, "layernorm", True), (5, 64, 5, 64)),
    (("forward", 3072, "layernorm", True), (5, 96, 4, 96)),
    (("forward", 8192, "rmsnorm", True), (5, 256, 4, 256)),
    (("forward", 16384, "rmsnorm", True), (5, 512, 4, 512)),
    (("backward", 384, "layernorm", False), (0, 16, 3, 256)),   # the bench step's backward
    (("backward", 256, "layernorm", False), (0, 8, 4, 256)),
    (("backward", 512, "layernorm", False), (0, 16, 4, 256)),
    (("backward", 1536, "rmsnorm", False), (6, 64, 3, 128)),     # two 64-thread groups
    (("backward", 1280, "layernorm", False), (7, 64, 3, 128)),
    (("backward", 2048, "layernorm", False), (3, 64, 4, 256)),     # row-group ring
    (("backward", 1024, "layernorm", False), (0, 32, 4, 256)),
    (("backward", 2560, "layernorm", False), (7, 128, 3, 256)),
    (("backward", 3072, "rmsnorm", False), (6, 128, 3, 256)),
    (("backward", 4096, "rmsnorm", False), (6, 128, 4, 256)),
    (("backward", 6144, "layernorm", False), (6, 256, 3, 512)),
    (("backward", 8192, "rmsnorm", False), (6, 256, 4, 512)),  # the second gate shape
    (("backward", 8192, "layernorm", False), (7, 512, 2, 512)),   # one 512-thread group
    (("backward", 7168, "layernorm", False), (8, 256, 4, 512)),
    (("backward", 8192, "layernorm", True), (7, 256, 4, 512)),
    (("backward", 8192, "rmsnorm", True), (7, 256, 4, 512)),
    (("backward", 12288, "layernorm", False), (8, 384, 4, 384)),  # one row group per CTA
    (("backward", 16384, "rmsnorm", False), (6, 512, 4, 512)),
    (("backward", 16384, "layernorm", False), (7, 512, 4, 512)),
    (("backward", 10240, "layernorm", True), (7, 320, 4, 320)),
    (("softmax", 384, "layernorm", False), (4, 16, 3, 256)),
    (("softmax", 256, "layernorm", False), (4, 8, 4, 256)),
    (("softmax", 2560, "layernorm", False), (5, 64, 5, 64)),
    (("softmax", 8192, "layernorm", False), (5, 256, 4, 256)),
    (("partials", 384, "layernorm", False), (4, 8, 6, 256)),
    (("partials", 8192, "layernorm", False), (5, 256, 4, 256)),
]


@pytest.mark.parametrize("args,want", EXPECTED, ids=lambda v: "-".join(map(str, v)))
def test_layout_of_measured_widths(args, want):
    direction, hidden, mode, option = args
    p = plan(direction, hidden, mode=mode, option=option)
    assert (p["kind"], p["group"], p["n"], p["block"]) == want, p


def test_persistent_backward_grids_fill_the_sms():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert plan("backward", 8192, mode="rmsnorm")["grid"] == sms       # one 512-thread CTA per SM
    assert plan("backward", 3072, mode="rmsnorm")["grid"] == 2 * sms   # two 256-thread CTAs


@pytest.mark.parametrize("dtype", [BF16, torch.float32])
@pytest.mark.parametrize("direction", ["forward", "backward", "softmax", "partials"])
def test_every_width_is_covered_by_whole_warps(direction, dtype):
    vec = 16 // torch.tensor([], dtype=dtype).element_size()
    top = 16384 if dtype == BF16 else 8192
    for hidden in range(vec, top + 1, vec):
        for mode in ("layernorm", "rmsnorm"):
            p = plan(direction, hidden, dtype=dtype, mode=mode, rows=4096)
            V = hidden // vec
            k, g, n, b = p["kind"], p["group"], p["n"], p["block"]
            assert b % 32 == 0 and 0 < b <= 512 and p["grid"] >= 1, (hidden, p)
            if k in (0, 4):       # lane groups: the row over g lanes, n vectors each
                assert g in (8, 16, 32) and g * n >= V and g * (n - 1) < V or n == 8, (hidden, p)
            elif k in (1, 3):     # pipelined CTA / row group
                assert g * n >= V, (hidden, p)
            elif k == 5:          # row-fitted CTA
                assert g == b and 64 <= b and b * n >= V and b * (n - 1) < V, (hidden, p)
            elif k in (6, 7, 8):  # one or two row groups of g threads
                assert b in (g, 2 * g) and g * n >= V, (hidden, p)
            else:
                assert k == 2, (hidden, p)
            if direction == "softmax":
                break             # softmax has no mode
