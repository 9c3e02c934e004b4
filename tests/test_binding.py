"""CPU checks of the Python binding's argument marshalling: the output dict keeps the caller's
tensors and allocates only the missing ones (with the documented shapes and dtypes), and the
per-call checks reject a wrong dtype, shape or device with a message naming the argument."""
import pytest

torch = pytest.importorskip("torch")

import manifold_constrained_hyper_mhc_gb300 as mhc  # noqa: E402


def test_outputs_keep_given_tensors_and_allocate_the_rest():
    T, H = 3, 64
    given = torch.zeros((T, H), dtype=torch.bfloat16)
    o = mhc._outputs(T, H, "cpu", {"layer_in": given}, True)
    assert o["layer_in"] is given
    assert set(o) == {"residual_out", "layer_in", "pre_mix", "post_mix", "comb_res_mix"}
    assert o["residual_out"].shape == (T, 4, H) and o["residual_out"].dtype == torch.bfloat16
    assert o["pre_mix"].shape == (T, 4) and o["pre_mix"].dtype == torch.float32
    assert o["post_mix"].shape == (T, 4) and o["post_mix"].dtype == torch.float32
    assert o["comb_res_mix"].shape == (T, 4, 4) and o["comb_res_mix"].dtype == torch.float32
    assert "residual_out" not in mhc._outputs(T, H, "cpu", None, False)


def test_outputs_allocate_nothing_when_all_are_given(monkeypatch):
    T, H = 2, 8
    full = {"residual_out": torch.empty((T, 4, H), dtype=torch.bfloat16),
            "layer_in": torch.empty((T, H), dtype=torch.bfloat16),
            "pre_mix": torch.empty((T, 4)), "post_mix": torch.empty((T, 4)), "comb_res_mix": torch.empty((T, 4, 4))}

    def no_alloc(*a, **k):
        raise AssertionError("allocated an output the caller supplied")

    monkeypatch.setattr(torch, "empty", no_alloc)
    o = mhc._outputs(T, H, "cpu", full, True)
    assert all(o[k] is full[k] for k in full)


def test_argument_checks_name_the_argument():
    with pytest.raises(TypeError, match="phi must be float32"):
        mhc._f32(torch.zeros((8, 24), dtype=torch.float64), "phi", (8, 24))
    with pytest.raises(ValueError, match=r"bias has shape \(23,\), expected \(24,\)"):
        mhc._f32(torch.zeros(23), "bias", (24,))
    with pytest.raises(TypeError, match="residual must be bfloat16"):
        mhc._bf16(torch.zeros((1, 4, 8)), "residual", (1, 4, 8))
    with pytest.raises(ValueError, match="layer_out must be a contiguous CUDA tensor"):
        mhc._bf16(torch.zeros((2, 8), dtype=torch.bfloat16), "layer_out", (2, 8))
    # the 16-bit bit patterns are accepted as bf16 (the shape is checked first)
    with pytest.raises(ValueError, match="CUDA"):
        mhc._bf16(torch.zeros((2, 8), dtype=torch.int16), "x", (2, 8))
