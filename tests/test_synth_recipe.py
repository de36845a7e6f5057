"""The seeded synthetic inputs follow the stated recipe.

synth/ is the one module the CUDA path and the oracle share: shapes, seeds and
value distributions, no arithmetic of the method.  These CPU tests check that
it is deterministic and that each workload's tensors have the shapes and the
value structure the input recipe states (outlier channels, per-channel
offsets, the centering bias, sink rows, rotary positions).
"""
import math

import pytest
import torch

import synth

# name -> (batch, layers, Hq, Hkv, D, stored context, io dtype)
SHAPES = {
    "tinygpt": (1, 1, 8, 8, 32, 260, torch.float32),
    "mlx8k": (1, 28, 24, 8, 128, 8192, torch.bfloat16),
    "q4_0_32k": (8, 32, 32, 8, 128, 32768, torch.bfloat16),
    "snapkv": (1, 1, 24, 8, 128, 512, torch.float16),
    "ring": (64, 32, 32, 8, 128, 4100, torch.bfloat16),
}


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_workload_shapes(name):
    w = synth.get_workload(name)
    B, L, Hq, Hkv, D, ctx, dt = SHAPES[name]
    assert (w.batch, w.layers, w.n_q_heads, w.n_kv_heads, w.head_dim, w.context) == (B, L, Hq, Hkv, D, ctx)
    assert synth.torch_dtype(w.io_dtype) == dt
    assert w.n_q_heads % w.n_kv_heads == 0 and w.group == Hq // Hkv


def test_streaming_and_snapkv_parameters():
    t = synth.get_workload("tinygpt")
    assert (t.layout, t.sink, t.window) == ("compact", 4, 256) and t.sink + t.window == t.context
    r = synth.get_workload("ring")
    assert (r.layout, r.sink, r.window, r.generated_steps) == ("ring", 4, 4096, 40000)
    assert (r.k_format, r.k_bits, r.v_format, r.v_bits, r.v_group) == ("kivi_chan", 4, "affine_token", 4, 32)
    s = synth.get_workload("snapkv")
    assert (s.prompt_len, s.obs_window, s.budget, s.n_sink, s.decode_steps) == (16384, 32, 512, 4, 256)
    m = synth.get_workload("mlx8k")
    assert (m.k_format, m.k_bits, m.k_group, m.v_format, m.v_bits, m.v_group) == \
        ("affine_token", 4, 64, "affine_token", 4, 64)
    q = synth.get_workload("q4_0_32k")
    assert (q.k_format, q.use_k_bias, q.v_format, q.v_bits, q.v_group) == ("q4_0", True, "affine_token", 8, 128)


def test_inputs_are_deterministic_and_windowed():
    w = synth.get_workload("mlx8k").with_(n_kv_heads=2, n_q_heads=6)
    k1, v1 = synth.layer_inputs(w, 3, 100, 40)
    k2, v2 = synth.layer_inputs(w, 3, 100, 40)
    assert torch.equal(k1, k2) and torch.equal(v1, v2)
    k3, _ = synth.layer_inputs(w, 4, 100, 40)
    assert not torch.equal(k1, k3)                    # layers differ
    q1, a1, b1 = synth.decode_token_inputs(w, 2, 7, 8199)
    q2, a2, b2 = synth.decode_token_inputs(w, 2, 7, 8199)
    assert torch.equal(q1, q2) and torch.equal(a1, a2) and torch.equal(b1, b2)
    assert q1.shape == (1, 6, 128) and a1.shape == (1, 2, 1, 128) and q1.dtype == torch.bfloat16


def test_outlier_channels_are_one_percent_scaled_by_ten():
    # 1% of the Hkv * D = 1024 (kv head, channel) key pairs, chosen per layer, scaled x10
    w = synth.get_workload("mlx8k")
    masks = [synth._outlier_mask(w, layer, "cpu") for layer in (0, 1)]
    for m in masks:
        assert m.shape == (8, 128)
        assert int((m == 10.0).sum()) == round(0.01 * 1024) and int((m == 1.0).sum()) == 1024 - 10
    assert not torch.equal(masks[0], masks[1])
    k, _ = synth.layer_inputs(w, 0, 0, 4096)
    std = k.float().std(dim=(0, 2))                   # per (kv head, channel)
    big = masks[0] == 10.0
    assert float(std[big].min()) > 6.0 and float(std[~big].max()) < 1.3


def test_channel_offsets_and_centering_bias_spreads():
    # per-(kv head, channel) K offset with standard deviation 2; centering bias with 1.5
    t = synth.get_workload("tinygpt").with_(n_kv_heads=64, n_q_heads=64)
    off = synth._channel_offsets(t, 0, "cpu")
    assert off.shape == (64, 32) and abs(float(off.std()) - 2.0) < 0.15
    q = synth.get_workload("q4_0_32k").with_(n_kv_heads=32, n_q_heads=128)
    kb = synth.k_bias(q, 0)
    assert kb.shape == (32, 128) and abs(float(kb.std()) - 1.5) < 0.1
    assert not torch.equal(kb, synth.k_bias(q, 1))   # one bias per layer
    # the keys carry that bias: their per-channel means sit on it
    k, _ = synth.layer_inputs(q.with_(batch=1), 0, 0, 2048)
    mean = k.float().mean(dim=(0, 2))
    assert float((mean - kb).abs().max()) < 0.15


def test_snapkv_sink_rows_scaled_by_eight():
    w = synth.get_workload("snapkv")
    k, _ = synth.snapkv_prefill(w, prompt_len=512)
    n = k.float().norm(dim=-1)                        # [1, Hkv, S]
    sink = n[..., :4].mean()
    rest = n[..., 4:].mean()
    assert 7.0 < float(sink / rest) < 9.0
    assert k.dtype == torch.float16 and k.shape == (1, 8, 512, 128)


def test_rope_is_a_rotation_at_absolute_positions():
    x = synth.normal((2, 3, 5, 128), 1, "rope")
    pos = torch.tensor([0, 1, 7, 4099, 40000])
    y = synth.rope_rotate(x, pos, 10000.0)
    torch.testing.assert_close(y.norm(dim=-1), x.norm(dim=-1), rtol=1e-5, atol=1e-5)
    torch.testing.assert_close(y[..., 0, :], x[..., 0, :])            # position 0: identity
    # relative property: <rope(a, i), rope(b, j)> depends only on i - j
    a, b = synth.normal((1, 1, 1, 128), 2, "a"), synth.normal((1, 1, 1, 128), 3, "b")
    def dot(i, j):
        ra = synth.rope_rotate(a, torch.tensor([i]), 10000.0)
        rb = synth.rope_rotate(b, torch.tensor([j]), 10000.0)
        return float((ra * rb).sum())
    assert math.isclose(dot(10, 3), dot(1010, 1003), rel_tol=1e-4, abs_tol=1e-4)
