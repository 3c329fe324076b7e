"""The tensor-core rate probes (rg_probe_mma_rate) run and report their work.

They are measurement tools beside the product path: each launch must finish
with status RG_OK (the tcgen05 probes' bounded wait did not expire) and report
the operation count its shape implies.  No timing is asserted here.
"""
import pytest
import torch

from tests.gpu_util import rg  # noqa: F401

pytestmark = pytest.mark.gpu


def test_probes_run_and_count_their_work(rg):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cases = [
        (rg.RG_PROBE_MMA_S8, 100, 0, 2.0 * 4 * sms * 8 * 100 * 8 * 16 * 8 * 32),
        (rg.RG_PROBE_MMA_S8, 10, 3, 2.0 * 3 * 8 * 10 * 8 * 16 * 8 * 32),
        (rg.RG_PROBE_TCGEN05_F16, 64, 0, 2.0 * sms * 64 * 4 * 128 * 256 * 16),
        (rg.RG_PROBE_TCGEN05_E4M3, 64, 0, 2.0 * sms * 64 * 4 * 128 * 256 * 32),
        (rg.RG_PROBE_TCGEN05_F16, 1, 1, 2.0 * 1 * 4 * 128 * 256 * 16),
        (rg.RG_PROBE_TCGEN05_F16_BMN, 64, 0, 2.0 * sms * 64 * 4 * 128 * 256 * 16),
        (rg.RG_PROBE_TCGEN05_F16_PAIR, 64, 0, 2.0 * (sms & ~1) * 64 * 4 * 128 * 256 * 16),
        (rg.RG_PROBE_TCGEN05_F16_PAIR_BMN, 64, 2, 2.0 * 2 * 64 * 4 * 128 * 256 * 16),
        (rg.RG_PROBE_TCGEN05_F16_PAIR_BMN_SYNC, 64, 0, 2.0 * (sms & ~1) * 64 * 4 * 128 * 256 * 16),
        (rg.RG_PROBE_MMA_F16, 100, 0, 2.0 * 4 * sms * 8 * 100 * 8 * 16 * 8 * 16),
    ]
    for kind, iters, blocks, want in cases:
        ops = rg.probe_mma_rate(kind, iters, blocks)
        assert ops == want
        torch.cuda.synchronize()
        assert rg.status() == rg.RG_OK


def test_probe_arguments_are_checked(rg):
    for kind, iters, blocks in ((8, 10, 0), (rg.RG_PROBE_MMA_S8, 0, 0), (rg.RG_PROBE_MMA_S8, 10, -1),
                                (rg.RG_PROBE_TCGEN05_F16_PAIR, 10, 3)):
        with pytest.raises(rg.ResGemmError) as e:
            rg.probe_mma_rate(kind, iters, blocks)
        assert e.value.code == rg.RG_ERR_ARG
