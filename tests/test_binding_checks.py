"""The Python binding's argument checks, on the CPU: dtype, shape and device
mismatches raise ValueError before anything is allocated or launched (the C
ABI sees only pointers and the sizes in moelora_dims, so these are the
binding's job)."""
import pytest
import torch

from lora_mixture_experts_gb300 import binding
from lora_mixture_experts_gb300.inputs import CONFIGS, make_moe_case


@pytest.fixture(scope="module")
def layer():
    return make_moe_case(CONFIGS["tiny"], seed=0, device="cpu")


def _fwd(d, **over):
    a = dict(d, **over)
    return binding.moe_lora_forward(a["x"], a["topk_ids"], a["topk_weights"], a["lora_ids"],
                                    a["W_gate_up"], a["W_down"], a["A_gu"], a["B_gu"], a["A_d"],
                                    a["B_d"], out=a.get("out"), ws=a.get("ws"))


@pytest.mark.parametrize("name,bad,match", [
    ("x", lambda d: d["x"].half(), "x: dtype"),
    ("topk_ids", lambda d: d["topk_ids"].long(), "topk_ids: dtype"),
    ("topk_weights", lambda d: d["topk_weights"].double(), "topk_weights: dtype"),
    ("topk_weights", lambda d: d["topk_weights"][:, :1].contiguous(), "topk_weights: shape"),
    ("lora_ids", lambda d: d["lora_ids"].long(), "lora_ids: dtype"),
    ("lora_ids", lambda d: d["lora_ids"][:-1].contiguous(), "lora_ids: shape"),
    ("W_down", lambda d: d["W_down"].transpose(1, 2).contiguous(), "W_down: shape"),
    ("A_gu", lambda d: d["A_gu"].float(), "A_gu: dtype"),
    ("B_d", lambda d: d["B_d"][:, :, :-8].contiguous(), "B_d: shape"),
    ("out", lambda d: torch.empty(d["x"].shape, dtype=torch.float32), "out: dtype"),
    ("ws", lambda d: torch.empty(1024, dtype=torch.int32), "ws: dtype"),
])
def test_forward_rejects_mismatched_tensors(lib, layer, name, bad, match):
    with pytest.raises(ValueError, match=match):
        _fwd(layer, **{name: bad(layer)})


def test_forward_requires_device_tensors(lib, layer):
    with pytest.raises(ValueError, match="device tensors"):
        _fwd(layer)


def test_linear_route_and_align_checks(lib):
    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    W = torch.zeros(32, 64, dtype=torch.bfloat16)
    lo = torch.zeros(4, dtype=torch.int32)
    with pytest.raises(ValueError, match="W: shape"):
        binding.moe_lora_linear(x, lo, W.t().contiguous())
    with pytest.raises(ValueError, match="lora_ids: dtype"):
        binding.moe_lora_linear(x, lo.long(), W)
    with pytest.raises(ValueError, match="logits: dtype"):
        binding.moe_lora_route(torch.zeros(4, 8, dtype=torch.float16), 2)
    with pytest.raises(ValueError, match="topk_ids: dtype"):
        binding.moe_lora_align(torch.zeros(4, 2, dtype=torch.int64), lo, 8, 1, 16)


class _OnDevice:
    """Stands in for a tensor on a CUDA device (there is none on this host):
    only the attributes the binding's checks read."""

    def __init__(self, index, shape, dtype):
        self.device = torch.device("cuda", index)
        self.shape = torch.Size(shape)
        self.dtype = dtype

    def dim(self):
        return len(self.shape)


class _Stream:
    def __init__(self, index):
        self.device = torch.device("cuda", index)


def test_tensors_off_the_current_device_are_rejected(lib, monkeypatch):
    # the library launches on the current device with the pointers it gets:
    # tensors of another device must raise before anything is launched
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 1)
    ids = _OnDevice(0, (4, 2), torch.int32)
    lo = _OnDevice(0, (4,), torch.int32)
    with pytest.raises(ValueError, match="current CUDA device is cuda:1"):
        binding.moe_lora_align(ids, lo, 8, 1, 16)
    with pytest.raises(ValueError, match="current CUDA device is cuda:1"):
        binding.moe_lora_align_noalloc(ids, lo, 8, 1, 16)
    with pytest.raises(ValueError, match="current CUDA device is cuda:1"):
        binding.moelora_get_error(_OnDevice(0, (64,), torch.uint8))


def test_stream_of_another_device_is_rejected(lib, monkeypatch):
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    ids = _OnDevice(0, (4, 2), torch.int32)
    lo = _OnDevice(0, (4,), torch.int32)
    with pytest.raises(ValueError, match="stream on cuda:1"):
        binding.moe_lora_align(ids, lo, 8, 1, 16, stream=_Stream(1))
