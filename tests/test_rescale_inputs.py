"""The planted-level inputs of ``rescale_cases`` take the online softmax's
rare branches (checked on the host from the exact scores of the rounded
inputs, no GPU): for DIFF V1 (both branches), DIFF V2 and Paired Head
Attention, rows past the first key tiles see a tile whose maximum rises more
than 8 log2 units above the running reference (the kernel rescales O), and
rows see tiles whose maximum rises by 4 to 8 (P above 2^4 under a stale
maximum).  Plain N(0, 1) inputs take neither: the contrast shows why the GPU
parity tests plant the levels."""
import numpy as np

import rescale_cases as rc
from differential_attention_causal_gb300 import inputs


def test_v1_planted_levels_take_both_branches():
    x = inputs.make_v1(inputs.V1Shape(1, 1024, 2, 64, 12, "bf16"), seed=1)
    rc.plant_v1(x, 64)
    for br in (0, 1):
        resc, stale = rc.v1_decisions(x, 0, 1, br)
        assert (resc[384:] > 0).all()            # every row past the third key tile rescales
        assert resc.max() >= 2 and stale.max() > 7.0


def test_v2_and_paired_planted_levels_take_both_branches():
    x = inputs.make_v2(inputs.V2Shape(1, 600, 4, 2, 128, "bf16"), seed=2)
    rc.plant_v2(x, 128)
    resc, stale = rc.v2_decisions(x, 0, 3, 2)
    assert (resc[384:] > 0).all() and stale.max() > 7.0
    x = inputs.make_paired(inputs.PairedShape(1, 400, 2, 64, "bf16"), seed=3)
    rc.plant_paired(x, 64)
    for head in (0, 1):
        resc, stale = rc.paired_decisions(x, 0, head)
        assert (resc[192:] > 0).all() and stale.max() > 7.0


def test_plain_random_inputs_never_rescale():
    x = inputs.make_v1(inputs.V1Shape(1, 1024, 1, 64, 12, "bf16"), seed=4)
    resc, stale = rc.v1_decisions(x, 0, 0, 0)
    assert resc.max() == 0 and stale.max() < 4.0
