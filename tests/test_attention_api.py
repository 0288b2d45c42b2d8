"""Host-side checks of the flash_attn_func-style entry points: options the
library does not provide are refused before any device work."""
import pytest
import torch

from exact_attention_93_gb300.attention import flash_attn_func, flash_attn_qkvpacked_func


def x():
    return torch.zeros(1, 128, 2, 64, dtype=torch.bfloat16)


def test_dropout_raises():
    with pytest.raises(NotImplementedError):
        flash_attn_func(x(), x(), x(), dropout_p=0.1)
    with pytest.raises(NotImplementedError):
        flash_attn_qkvpacked_func(torch.zeros(1, 128, 3, 2, 64, dtype=torch.bfloat16),
                                  dropout_p=0.1)


@pytest.mark.parametrize("kw", [{"window_size": (-2, 0)}, {"window_size": (3, -5)},
                                {"alibi_slopes": torch.ones(3)},
                                {"alibi_slopes": torch.ones(2, 2)}])
def test_bad_window_or_slope_shapes_raise(kw):
    with pytest.raises(ValueError):
        flash_attn_func(x(), x(), x(), **kw)


def test_packed_shape_is_checked():
    with pytest.raises(ValueError):
        flash_attn_qkvpacked_func(torch.zeros(1, 128, 2, 2, 64, dtype=torch.bfloat16))


def test_cpu_tensors_are_refused():
    with pytest.raises(ValueError):
        flash_attn_func(x(), x(), x())


def test_block_mask_shape_is_checked():
    with pytest.raises(ValueError):
        flash_attn_func(x(), x(), x(), block_mask=torch.ones(2, 2, dtype=torch.uint8))
