"""The measured ceilings the bench divides by: the instruction probes (IMMA, FFMA) and the HBM
probes (16-byte stores, loads and a copy over a buffer far larger than the L2).  The bounds are
wide: they catch a probe that times nothing (far above the hardware) or that is broken (far below),
not a slow or throttled GPU."""
import pytest
import torch

import software_pipelined_tiled_pipeline_gb300 as gp

pytestmark = pytest.mark.gpu


def test_instruction_probes_are_plausible():
    s = torch.cuda.current_stream()
    imma = gp.probe_peak("imma_s8", s)
    ffma = gp.probe_peak("ffma_f32", s)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # FFMA: at most 128 lanes x 2 FLOP per SM per cycle at 3 GHz; at least a tenth of that at 1 GHz
    assert sms * 128 * 2 * 1e9 / 10 < ffma < sms * 128 * 2 * 3e9
    assert 1e13 < imma < 1e15


def test_hbm_probes_are_plausible_and_leave_the_copy_in_place():
    buf = torch.zeros(1 << 30, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    rates = {k: gp.probe_hbm(k, buf, s) for k in ("write", "read", "copy")}
    for k, r in rates.items():
        assert 1e12 < r < 2e13, (k, r)
    torch.cuda.synchronize()
    # the copy probe moves the first half onto the second
    half = buf.numel() // 2
    assert torch.equal(buf[:half], buf[half:])
    with pytest.raises(gp.GemmError):
        gp.probe_hbm("read", buf[:1024], s)
