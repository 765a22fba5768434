"""moe_convert_bf16_to_f16, the load-time step that makes the fp16 down
weights: against torch's own bf16 -> fp16 cast (round to nearest even) over
every finite bf16 bit pattern, ragged lengths, and the range check."""
import pytest
import torch

from sparse_moe_ffn_gb300 import binding

pytestmark = pytest.mark.gpu
MOE_ERR_DEVICE_CHECK = 5


def test_every_bf16_value_matches_torch_cast():
    bits = torch.arange(1 << 16, dtype=torch.int32).to(torch.int16)
    v = bits.view(torch.bfloat16)
    v = v[torch.isfinite(v.float()) & (v.float().abs() <= 65504)].contiguous().cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = binding.convert_bf16_to_f16(v, status=status)
    assert torch.equal(got.view(torch.int16), v.to(torch.float16).view(torch.int16))
    assert int(status.item()) == 0


@pytest.mark.parametrize("n", [1, 7, 8, 9, 4096 + 5, 3 * 1024 * 1024 + 3])
def test_ragged_lengths(n):
    x = (0.02 * torch.randn(n, generator=torch.Generator().manual_seed(n))).to(torch.bfloat16).cuda()
    assert torch.equal(binding.convert_bf16_to_f16(x), x.to(torch.float16))


def test_out_of_range_is_reported():
    x = torch.zeros(24, dtype=torch.bfloat16)
    x[13] = 65536.0  # the first bf16 value above fp16's range
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.convert_bf16_to_f16(x.cuda(), status=status)
    assert int(status.item()) == MOE_ERR_DEVICE_CHECK
    with pytest.raises(binding.MoEError):
        binding.prepare_weights({"w_down": x.cuda().view(1, 24, 1)})
