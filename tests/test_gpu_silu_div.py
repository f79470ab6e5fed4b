"""The L1 epilogue's SiLU division (branch-free Newton-Raphson reciprocal with
Markstein's residual correction) against the IEEE operations of this GPU."""
import pytest

pytestmark = pytest.mark.gpu


def test_silu_division_matches_ieee_division():
    import torch
    import moe_expert_layer_scan_gb300 as mm
    counts = torch.zeros(5, dtype=torch.int64, device="cuda")
    pairs = 1 << 28
    mm.mm_debug_div_check(pairs, 0x5EED, counts.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    rcp_bad, normal_bad, tiny_bad, checked, far = (int(v) for v in counts.cpu())
    assert checked == pairs
    assert rcp_bad == 0       # every refined reciprocal is the correctly rounded one
    assert normal_bad == 0    # so every normal quotient equals IEEE division
    assert far == 0           # and no quotient is more than one unit in the last place away
    print(f"subnormal or zero quotients differing in the last place: {tiny_bad} of {pairs}")
