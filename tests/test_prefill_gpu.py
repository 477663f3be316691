"""Causal GQA prefill (K1 + K2) on the GPU against the fp64 oracle, via the C ABI."""
import pytest
import torch

import oracle
from qwen3_qk_norm_gb300 import binding, inputs
from qwen3_qk_norm_gb300.inputs import WORKLOADS
from gpu_util import assert_close_attention, assert_within_one_ulp

pytestmark = pytest.mark.gpu


def run_prefill(x, theta, eps=1e-6):
    d = {k: t.cuda() for k, t in x.items()}
    out = binding.prefill(d["q"], d["k"], d["v"], d["q_gamma"], d["k_gamma"], theta, eps)
    torch.cuda.synchronize()
    return out


# small shapes: several M tiles and KV tiles, ragged tails, every g
@pytest.mark.parametrize("B,T,Hq,Hkv,theta", [
    (1, 1, 16, 8, 1e6),      # a single token
    (1, 2, 4, 4, 1e6),       # g = 1
    (1, 127, 8, 4, 1e6),     # one KV tile minus one
    (2, 129, 16, 8, 1e6),    # one KV tile plus one, B > 1
    (1, 255, 8, 1, 1e7),     # g = 8
    (1, 300, 16, 1, 1e6),    # g = 16
    (2, 200, 2, 2, 1e6),     # g = 1, ragged
    (3, 520, 8, 2, 1e6),     # g = 4, five KV tiles
])
def test_prefill_small_shapes(cuda_lib, B, T, Hq, Hkv, theta):
    x = inputs.prefill_inputs(B, T, Hq, Hkv, seed=B * 1000 + T)
    ref = oracle.prefill(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], theta, 1e-6)
    assert_close_attention(run_prefill(x, theta), ref, f"prefill B{B} T{T} Hq{Hq} Hkv{Hkv}")


def test_prefill_qwen3_06b_t128_full(cuda_lib):
    w = WORKLOADS["qwen3-0.6b-prefill-b1-t128"]
    x = inputs.workload_inputs(w)
    ref = oracle.prefill(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], w.theta, w.eps)
    assert_close_attention(run_prefill(x, w.theta), ref, w.name)


def test_prefill_with_norm_outliers(cuda_lib):
    x = inputs.prefill_inputs(1, 700, 32, 8, seed=5, outlier_frac=0.01, outlier_scale=30.0)
    ref = oracle.prefill(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    assert_close_attention(run_prefill(x, 1e6), ref, "outliers")


@pytest.mark.parametrize("gmax", [1.0, 1.9, 2.1, 2.3])  # bound 16, 59 | 72, 86 (log2 units)
def test_prefill_both_softmax_paths(cuda_lib, gmax):
    """QK-Norm bounds the logits by sqrt(128) max|gamma_q| max|gamma_k|. Small
    gammas take the fixed-shift softmax; large ones (bound above the kernel's
    limit) take the online-max path. Both must match the oracle."""
    x = inputs.prefill_inputs(1, 300, 16, 4, seed=int(gmax * 10))
    g = torch.Generator().manual_seed(77)
    x["q_gamma"] = (torch.rand(128, generator=g) * gmax).to(torch.bfloat16)
    x["k_gamma"] = (torch.rand(128, generator=g) * gmax).to(torch.bfloat16)
    ref = oracle.prefill(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    assert_close_attention(run_prefill(x, 1e6), ref, f"gamma max {gmax}")


@pytest.mark.parametrize("gmax", [2.5, 6.0])  # bound 102, 587 (log2 units): online max
def test_prefill_large_gamma_against_the_bf16_rounded_oracle(cuda_lib, gmax):
    """Above gamma 2.3 the bf16 rounding of qhat and khat alone moves the exact
    output by more than the tolerance (tests/test_oracle_rounding_pins.py), so
    the kernels, whose products take bf16 qhat and khat, are compared with the
    oracle that rounds them the same way (once, after RoPE) and computes
    everything else in fp64."""
    x = inputs.prefill_inputs(1, 300, 16, 4, seed=int(gmax * 10))
    g = torch.Generator().manual_seed(77)
    x["q_gamma"] = (torch.rand(128, generator=g) * gmax).to(torch.bfloat16)
    x["k_gamma"] = (torch.rand(128, generator=g) * gmax).to(torch.bfloat16)
    ref = oracle.prefill_rounded(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6, 1)
    assert_close_attention(run_prefill(x, 1e6), ref, f"gamma max {gmax}, bf16-rounded oracle")


def test_prefill_future_tokens_leave_past_rows_bit_identical(cuda_lib):
    B, T, Hq, Hkv, cut = 1, 400, 8, 2, 170
    x = inputs.prefill_inputs(B, T, Hq, Hkv, seed=9)
    a = run_prefill(x, 1e6)
    y = dict(x)
    y["k"] = x["k"].clone()
    y["v"] = x["v"].clone()
    y["k"][:, cut:] = inputs.prefill_inputs(B, T - cut, Hkv, Hkv, seed=10)["k"]
    y["v"][:, cut:] = inputs.prefill_inputs(B, T - cut, Hkv, Hkv, seed=11)["v"]
    b = run_prefill(y, 1e6)
    assert torch.equal(a[:, :cut], b[:, :cut])
    assert not torch.equal(a[:, cut:], b[:, cut:])


def test_prefill_row0_is_v_row0(cuda_lib):
    """Row 0 sees only key 0, so it returns V row 0: up to the bf16 rounding of
    its single weight and of the output (one bf16 ulp)."""
    x = inputs.prefill_inputs(2, 64, 16, 4, seed=12)
    out = run_prefill(x, 1e6).cpu()
    for h in range(16):
        assert_within_one_ulp(out[:, 0, h], x["v"][:, 0, h // 4].double(), "row 0")


def test_prefill_halves_equal_the_whole_call(cuda_lib):
    """q3a_prefill_prologue (keys) then q3a_prefill_attention (query norm and
    attention) on one workspace give q3a_prefill's bits."""
    B, T, Hq, Hkv = 2, 333, 16, 4
    x = {k: t.cuda() for k, t in inputs.prefill_inputs(B, T, Hq, Hkv, seed=16).items()}
    whole = binding.prefill(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    ws = torch.empty(binding.prefill_workspace_size(B, T, Hq, Hkv), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty_like(x["q"])
    binding.prefill_prologue(x["k"], x["q_gamma"], x["k_gamma"], Hq, 1e6, 1e-6, ws)
    binding.prefill_attention(x["q"], x["v"], x["q_gamma"], out, 1e-6, ws)
    torch.cuda.synchronize()
    assert torch.equal(out, whole)


def test_prefill_output_only_16_byte_aligned(cuda_lib):
    """The contract asks for 16-byte aligned tensors; the kernel writes 32-byte
    pieces of each output row when it can and 16-byte ones otherwise: an
    output that starts 16 bytes into a buffer gets the same bits."""
    B, T, Hq, Hkv = 1, 200, 16, 4
    x = {k: t.cuda() for k, t in inputs.prefill_inputs(B, T, Hq, Hkv, seed=17).items()}
    full = binding.prefill(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    buf = torch.empty(B * T * Hq * 128 + 8, dtype=torch.bfloat16, device="cuda")
    out = buf[8:].view(B, T, Hq, 128)
    assert out.data_ptr() % 32 == 16
    binding.prefill(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6, out=out)
    torch.cuda.synchronize()
    assert torch.equal(out, full)


def test_prefill_is_deterministic(cuda_lib):
    x = inputs.prefill_inputs(1, 300, 32, 8, seed=13)
    assert torch.equal(run_prefill(x, 1e6), run_prefill(x, 1e6))


def test_prefill_rejects_bad_group_and_leaves_out_untouched(cuda_lib):
    x = {k: t.cuda() for k, t in inputs.prefill_inputs(1, 8, 12, 8, seed=14).items()}
    out = torch.full_like(x["q"], 7.0)
    with pytest.raises(binding.Q3AError) as e:
        binding.prefill(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6, out=out)
    assert e.value.status == binding.Q3A_EINVAL
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())


def test_prefill_no_device_error_word(cuda_lib):
    x = {k: t.cuda() for k, t in inputs.prefill_inputs(1, 130, 8, 2, seed=15).items()}
    ws = torch.empty(binding.prefill_workspace_size(1, 130, 8, 2), dtype=torch.uint8,
                     device="cuda")
    binding.prefill(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6, workspace=ws)
    assert binding.last_device_error(ws) == binding.Q3A_OK


def test_prefill_more_items_than_ctas_full_parity(cuda_lib):
    """160 work items (pairs of 32-token Q tiles of 8 KV groups) on a GPU with
    fewer SMs than that: some persistent CTAs take a second item in the snake
    order's partial last round. Every output row against the oracle."""
    B, T, Hq, Hkv = 2, 1280, 32, 4
    x = inputs.prefill_inputs(B, T, Hq, Hkv, seed=31)
    ref = oracle.prefill(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    assert_close_attention(run_prefill(x, 1e6), ref, "160 items")
