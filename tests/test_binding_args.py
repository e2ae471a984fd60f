"""The Python binding's argument checks (no GPU): malformed tensors are refused before any call into
the library, and a planning handle refuses to run at all."""
import types

import pytest
import torch

import complexity_matmul_gb300 as lcg

STREAM = types.SimpleNamespace(cuda_stream=0)     # stands in for a CUDA stream; never used by a launch


@pytest.fixture()
def h():
    handle = lcg.Handle(lcg.PLANNING_DEVICE)
    yield handle
    handle.close()


def _t(*shape, dtype=torch.bfloat16):
    return torch.zeros(*shape, dtype=dtype)


def test_k_mismatch(h):
    with pytest.raises(ValueError):
        h.run(_t(16, 64), _t(32, 48), stream=STREAM)


def test_dtype_mismatch(h):
    with pytest.raises(TypeError):
        h.run(_t(16, 64), _t(32, 64, dtype=torch.float16), stream=STREAM)


def test_unsupported_dtype(h):
    with pytest.raises(TypeError):
        h.run(_t(16, 64, dtype=torch.float32), _t(32, 64, dtype=torch.float32), stream=STREAM)


def test_strided_k_refused(h):
    with pytest.raises(ValueError):
        h.run(_t(64, 16).t(), _t(32, 64), stream=STREAM)


def test_wrong_output_shape(h):
    with pytest.raises(ValueError):
        h.run(_t(16, 64), _t(32, 64), C=_t(16, 31), stream=STREAM)


def test_bias_and_residual_shapes(h):
    with pytest.raises(ValueError):
        h.run(_t(16, 64), _t(32, 64), C=_t(16, 32), stream=STREAM, bias=_t(31))
    with pytest.raises(ValueError):
        h.run(_t(16, 64), _t(32, 64), C=_t(16, 32), stream=STREAM, residual=_t(16, 33))


def test_planning_handle_refuses_to_run(h):
    with pytest.raises(lcg.LcgemmError) as e:
        h.run(_t(16, 64), _t(32, 64), C=_t(16, 32), stream=STREAM)
    assert e.value.code == lcg.ERR_ARG
