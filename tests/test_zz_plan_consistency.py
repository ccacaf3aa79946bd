"""The host-only plan queries predict the plans of actual launches on this
device (GPU; collected late so that they run after the parity tests)."""
import pytest

import synth

pytestmark = pytest.mark.gpu


def test_plan_query_matches_the_launch():
    """The host-only plan query predicts the plan of an actual call on this device."""
    import torch
    import quantized_gemm_tma_gb300 as hq
    from gpu_helpers import DevWeight, run_gemm
    props = torch.cuda.get_device_properties(0)
    optin = getattr(props, "shared_memory_per_block_optin", 232448)
    for seed, m, n, k in ((11, 16, 512, 1024), (12, 300, 256, 512), (13, 64, 8192, 256)):
        qw, acts = synth.dense_w4a16_asym(seed, m, n, k)
        dw = DevWeight(qw)
        run_gemm(dw, acts)
        assert hq.hq_last_plan() == hq.hq_plan_query(dw.desc, m, "bf16", props.multi_processor_count, optin)


def test_moe_plan_query_matches_the_launch():
    import torch
    import quantized_gemm_tma_gb300 as hq
    from gpu_helpers import DevWeight, run_moe
    props = torch.cuda.get_device_properties(0)
    optin = getattr(props, "shared_memory_per_block_optin", 232448)
    for seed, t, e, n, k, topk in ((30, 24, 8, 256, 256, 2), (31, 300, 4, 256, 256, 4)):
        qw, acts, r = synth.moe_mxfp4(seed, t, num_experts=e, n=n, k=k, topk=topk)
        dw = DevWeight(qw)
        y, st = run_moe(dw, acts, r)
        assert st == 0
        assert hq.hq_last_plan() == hq.hq_moe_plan_query(dw.desc, t, topk, props.multi_processor_count, optin)
