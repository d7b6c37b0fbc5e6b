"""Host-side checks of the Python binding that need no GPU."""
import types

import pytest


class _Dev:
    """Stand-in for a CUDA tensor: only its device index matters here."""

    def __init__(self, index):
        self.index = index

    def get_device(self):
        return self.index


def test_tensors_must_share_the_metadata_device():
    import expand_gemm_gb300 as eg
    meta = types.SimpleNamespace(no_lora_flag=_Dev(0))
    eg._same_device(meta, [("x", _Dev(0)), ("bias", None), ("y", _Dev(0))])
    with pytest.raises(ValueError, match="y is on cuda:1, the metadata on cuda:0"):
        eg._same_device(meta, [("x", _Dev(0)), ("y", _Dev(1))])


def test_no_cpu_path():
    """CPU tensors are refused before anything reaches the library."""
    import torch
    import expand_gemm_gb300 as eg
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        eg._need(torch.zeros(4, dtype=torch.int32), "token_lora_mapping", torch.int32)
