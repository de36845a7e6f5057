"""Host-side checks of the C-ABI library: it loads, exports every function the
header declares, and its argument validation and plane layout behave as the
header states.  No call here touches a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "bit_kv_cache_quant_gb300", "libkvq.so")


@pytest.fixture(scope="module")
def kvq():
    if not os.path.exists(LIB):
        import __graft_entry__

        __graft_entry__.build()
    import bit_kv_cache_quant_gb300 as m

    return m


def test_exports_every_declared_function(kvq):
    names = kvq.declared_functions()
    assert len(names) >= 15
    raw = ctypes.CDLL(kvq.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), f"{n} declared in kvq.h but not exported"
    assert kvq.lib.kvq_abi_version() == 2


def test_header_functions_are_extern_c():
    with open(os.path.join(ROOT, "include", "kvq.h")) as f:
        text = f.read()
    assert 'extern "C"' in text
    # every declaration is a plain C signature: no torch, no C++ references
    assert "torch" not in text.replace("torch types", "") and "&" not in re.sub(r"/\*.*?\*/", "", text, flags=re.S)


def _cfg(kvq, **kw):
    base = dict(batch=2, n_kv_heads=4, head_dim=128, capacity=100, k_format="affine_token", k_bits=4, k_group=64,
                v_format="affine_token", v_bits=4, v_group=64)
    base.update(kw)
    bias = base.pop("k_bias", None)
    cfg = kvq.make_config(**base)
    if bias is not None:
        cfg.k_bias = bias
    return cfg


def _status(kvq, cfg):
    lay = kvq.kvq_cache_layout()
    return kvq.lib.kvq_cache_layout_query(ctypes.byref(cfg), ctypes.byref(lay)), lay


def test_layout_planes_are_aligned_and_sized(kvq):
    st, lay = _status(kvq, _cfg(kvq))
    assert st == 0
    assert lay.cap_alloc == 128 and lay.k_row_bytes == 64 and lay.k_n_groups == 2
    offs = [lay.state, lay.split_sem, lay.k_codes, lay.k_tok_scale, lay.k_tok_zero, lay.v_codes, lay.v_tok_scale,
            lay.v_tok_zero]
    assert all(o % 256 == 0 for o in offs) and offs == sorted(offs)
    assert lay.k_tok_scale - lay.k_codes >= 2 * 4 * 128 * 64
    assert lay.total_bytes >= lay.v_tok_zero + 2 * 4 * 128 * 2 * 2
    assert lay.k_ch_scale == 0 and lay.k_bias == 0


def test_layout_matches_byte_accounting(kvq):
    # codes + metadata per stored row agree with the oracle's bytes-per-token rule
    from oracle import accounting as acc

    for fmt, bits, group in (("affine_token", 4, 64), ("affine_token", 8, 128), ("q4_0", 4, 32), ("fp16", 16, 0)):
        vfmt = "fp16" if fmt in ("fp16", "q4_0") else fmt
        cfg = _cfg(kvq, k_format=fmt, k_bits=bits, k_group=group, v_format=vfmt, v_bits=bits if vfmt != "fp16" else 16,
                   v_group=group if vfmt != "fp16" else 0)
        st, lay = _status(kvq, cfg)
        assert st == 0, kvq.lib.kvq_last_error()
        meta = lay.k_n_groups * 2 * (2 if fmt == "affine_token" else 1)
        assert lay.k_row_bytes + meta == acc.side_bytes_per_token(fmt, bits, group, 128)


@pytest.mark.parametrize("bad,code", [
    (dict(head_dim=96), 2),
    (dict(batch=0), 1),
    (dict(k_format="kivi_chan", k_bits=3), 1),
    (dict(k_group=48), 1),
    (dict(v_format="q4_0", v_bits=4, v_group=32), 2),
    (dict(v_format="kivi_chan", v_bits=8, v_group=0), 2),
    (dict(layout="compact", sink=4, window=96), 1),       # capacity < sink + window + 1
    (dict(layout="ring", sink=4, window=200), 1),
    (dict(layout="ring", sink=4, window=0), 1),
])
def test_invalid_configs_rejected(kvq, bad, code):
    st, _ = _status(kvq, _cfg(kvq, **bad))
    assert st == code, kvq.lib.kvq_last_error()
    assert kvq.lib.kvq_last_error()


def test_bias_gate(kvq):
    # a mean-centering bias with non-Q4_0 keys is rejected before any device work
    st, _ = _status(kvq, _cfg(kvq, k_bias=0x1000))
    assert st == 2 and b"Q4_0" in kvq.lib.kvq_last_error()
    st, lay = _status(kvq, _cfg(kvq, k_format="q4_0", k_bits=4, k_group=32, k_bias=0x1000))
    assert st == 0 and lay.k_bias != 0


def test_snapkv_argument_checks(kvq):
    f = kvq.lib.snapkv_select
    ws = kvq.snapkv_workspace_bytes(1, 8, 16384, 128, 32)
    assert ws >= 8 * 16384 * 4
    # n_sink > budget, bad head_dim, window out of range: all rejected on the host
    assert f(0x1000, 100, 1, 1, 100, 128, 32, 4, 5, None, 0x2000, 0x3000, ws, None) == 1
    assert f(0x1000, 100, 1, 1, 100, 96, 32, 8, 4, None, 0x2000, 0x3000, ws, None) == 2
    assert f(0x1000, 100, 1, 1, 100, 128, 65, 8, 4, None, 0x2000, 0x3000, ws, None) == 2
    assert kvq.lib.snapkv_topk(0x1000, 1, 1, 10, 3, 4, 0x2000, None) == 1


def test_null_handles(kvq):
    assert kvq.lib.kvq_append(None, None, None, 1, 1, 0, None) == 1
    assert kvq.lib.kvq_decode_attn(None, None, None, 1, 1, 0.0, None, 0, None) == 1
    assert kvq.lib.kvq_decode_workspace_bytes(None, 8) == 0


def test_residual_buffer_layout(kvq):
    # KIVI_BLOCK keys: per-block channel metadata [B][Hkv][cap_alloc / R][D] fp16 and fp32 tails [B][Hkv][R][D]
    cfg = _cfg(kvq, capacity=300, k_format="kivi_block", k_bits=4, k_group=128, v_format="affine_token", v_bits=4,
               v_group=32)
    st, lay = _status(kvq, cfg)
    assert st == 0, kvq.lib.kvq_last_error()
    assert lay.cap_alloc == 320 and lay.k_n_groups == 0 and lay.k_tok_scale == 0
    BH, D = 2 * 4, 128
    offs = [lay.k_codes, lay.k_blk_scale, lay.k_blk_zero, lay.k_tail, lay.v_tail]
    assert all(o and o % 256 == 0 for o in offs) and offs == sorted(offs)
    assert lay.k_blk_zero - lay.k_blk_scale >= BH * (320 // 128) * D * 2
    assert lay.v_tail - lay.k_tail >= BH * 128 * D * 4 and lay.total_bytes >= lay.v_tail + BH * 128 * D * 4
    st, lay = _status(kvq, _cfg(kvq))
    assert lay.k_blk_scale == 0 and lay.k_tail == 0 and lay.v_tail == 0


@pytest.mark.parametrize("bad,code", [
    (dict(k_group=32), 2),                                           # block length not 64 or 128
    (dict(k_bits=2), 1),
    (dict(layout="compact", sink=4, window=64, capacity=200), 2),   # residual buffers are LINEAR
    (dict(v_format="fp16", v_bits=16, v_group=0), 2),                # values must be AFFINE_TOKEN
    (dict(capacity=100), 2),                                         # capacity below one block
    (dict(v_format="kivi_block", v_bits=4, v_group=64), 2),          # a K-side format
])
def test_residual_buffer_invalid_configs(kvq, bad, code):
    base = dict(capacity=256, k_format="kivi_block", k_bits=4, k_group=128, v_format="affine_token", v_bits=4,
                v_group=32)
    base.update(bad)
    st, _ = _status(kvq, _cfg(kvq, **base))
    assert st == code, kvq.lib.kvq_last_error()


def test_row_count_limit(kvq):
    # each code plane is one tensor of B * Hkv * cap_alloc rows addressed with a
    # signed 32-bit row coordinate: 2^31 - 64 rows or more are refused up front
    st, _ = _status(kvq, _cfg(kvq, batch=1 << 16, n_kv_heads=8, capacity=4096))
    assert st == 2 and b"2^31" in kvq.lib.kvq_last_error()
    st, _ = _status(kvq, _cfg(kvq, batch=1, n_kv_heads=1, capacity=(1 << 31) - 1))
    assert st == 2
    # batch * n_kv_heads * capacity near 2^93 must not wrap around into an accepted size
    st, _ = _status(kvq, _cfg(kvq, batch=(1 << 31) - 1, n_kv_heads=(1 << 31) - 1, capacity=(1 << 31) - 64))
    assert st == 2
    st, lay = _status(kvq, _cfg(kvq, batch=8, n_kv_heads=8, capacity=(1 << 25) - 64))
    assert st == 0, kvq.lib.kvq_last_error()
    assert lay.cap_alloc == (1 << 25) - 64
    assert lay.total_bytes > 64 * ((1 << 25) - 64) * 64 * 2      # ~256 GB of 4-bit K and V codes


def test_binding_checks_shapes_before_any_call(kvq):
    # the C entry points get raw pointers and cannot see shapes or dtypes; the
    # binding refuses mismatched tensors before calling them
    import torch

    c = object.__new__(kvq.KVCache)
    c.batch, c.n_kv_heads, c.head_dim, c.handle, c.launches, c._ws = 2, 4, 64, None, 0, {}
    k = torch.zeros((2, 4, 3, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="must match"):
        c.append(k, k.float())
    with pytest.raises(ValueError, match="must match"):
        c.append(k, k[:, :, :2])
    with pytest.raises(ValueError, match=r"\[2, 4, n, 64\]"):
        c.append(k[:, :3].contiguous(), k[:, :3].contiguous())
    with pytest.raises(ValueError, match="unsupported input dtype"):
        c.append(k.to(torch.int8), k.to(torch.int8))
    with pytest.raises(ValueError, match="n_tokens"):
        c.convert(k, k, 4)
    with pytest.raises(ValueError, match="q must be"):
        c.decode_attn(torch.zeros((2, 8, 32), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="out must"):
        q = torch.zeros((2, 8, 64), dtype=torch.bfloat16)
        c.decode_attn(q, out=torch.zeros((2, 8, 64), dtype=torch.float32))
    with pytest.raises(ValueError, match="CUDA tensor"):
        c.append(k, k)


def test_readme_c_example_compiles_and_links(kvq, tmp_path):
    # the README's C example is written against this header and this library
    import re
    import shutil
    import subprocess

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    with open(os.path.join(ROOT, "README.md")) as f:
        code = re.search(r"```c\n(.*?)```", f.read(), re.S).group(1)
    src = tmp_path / "example.c"
    src.write_text(code)
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    cuda_lib = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "lib64")
    obj = tmp_path / "example.o"
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-fPIC", "-c", str(src), "-o", str(obj),
                        "-I", os.path.join(ROOT, "include"), "-I", cuda_inc], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([gcc, "-shared", "-Wl,--no-undefined", "-o", str(tmp_path / "example.so"), str(obj),
                        "-L", os.path.dirname(kvq.LIB_PATH), "-lkvq", "-L", cuda_lib, "-lcudart"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


# GB300: 152 SMs.  Tensor-core decode: eight-warp CTAs, two per SM (one with
# over four query heads per kv head), when the grid fits one wave, or one
# sixteen-warp CTA per SM (wide 2) when up to four heads per kv head leave
# every (b, kv head) at least two splits of four tiles; otherwise four-warp
# CTAs, four per SM (eight-warp, two per SM, over four heads), over two whole
# waves.  At most 128 splits per (b, kv head).
SMS = 152


def _plan(kvq, n_q_heads, sms=SMS, **cfg):
    return kvq.kvq_decode_plan_query(_cfg(kvq, **cfg), n_q_heads, sms)


def test_decode_plan_of_the_workloads(kvq):
    # 8K mlx layer (B1, 8 kv heads, G 3): 19 splits, 152 sixteen-warp CTAs, one per SM
    assert _plan(kvq, 24, batch=1, n_kv_heads=8, capacity=8192 + 64) == (32, 19, 2)
    # the same layer with a KIVI residual buffer: one split fewer for the tail CTA (160 - 8 = 152 CTAs)
    assert _plan(kvq, 24, batch=1, n_kv_heads=8, capacity=8192 + 128, k_format="kivi_block", k_bits=4,
                 k_group=128, v_group=32) == (32, 18, 2)
    # over four heads per kv head: eight-warp CTAs over two head groups, one per SM, in two waves
    assert _plan(kvq, 48, batch=1, n_kv_heads=8, capacity=8192 + 64)[2] == 0
    # SnapKV's kept cache (768 rows): three splits of four tiles, sixteen-warp CTAs
    assert _plan(kvq, 24, batch=1, n_kv_heads=8, capacity=768, k_format="fp16", k_bits=16, k_group=0,
                 v_format="fp16", v_bits=16, v_group=0) == (12, 3, 2)
    # a 300-row cache has no two splits of four tiles: eight-warp CTAs, four splits
    assert _plan(kvq, 24, batch=2, n_kv_heads=4, capacity=300) == (4, 4, 1)
    # 32K Q4_0 layer (B8, 8 kv heads, G 4): 19 splits, 1216 four-warp CTAs = two whole waves of 4 per SM
    ns, ntc, wide = _plan(kvq, 32, batch=8, n_kv_heads=8, capacity=32768 + 64, k_format="q4_0", k_group=32,
                          v_bits=8, v_group=128)
    assert (ntc, wide) == (19, 0) and 64 * ntc == 2 * 4 * SMS
    # ring 4 + 4096 (B64, 8 kv heads, G 4): 2 splits, 1024 CTAs inside two waves
    ns, ntc, wide = _plan(kvq, 32, batch=64, n_kv_heads=8, capacity=4100, layout="ring", sink=4, window=4096,
                          k_format="kivi_chan", k_bits=4, k_group=0, v_group=32)
    assert (ntc, wide) == (2, 0)
    # tinygpt (D 32, fp32: the CUDA-core kernel): 261 rows over 4 splits of at least 64
    ns, _, _ = _plan(kvq, 8, batch=1, n_kv_heads=8, head_dim=32, capacity=261, layout="compact", sink=4,
                     window=256, k_format="kivi_chan", k_bits=8, k_group=0, v_bits=8, v_group=32)
    assert ns == 4


@pytest.mark.parametrize("sms", [SMS, 148, 132])
def test_decode_plan_invariants(kvq, sms):
    for B, H, cap, G in [(1, 8, 8256, 3), (1, 8, 8256, 8), (2, 4, 1000, 2), (8, 8, 32832, 4), (64, 8, 4100, 4),
                         (1, 1, 64, 1), (1, 2, 300000, 6), (16, 8, 131072, 5), (4, 8, 5000, 7)]:
        ns, ntc, wide = _plan(kvq, G * H, sms=sms, batch=B, n_kv_heads=H, capacity=cap)
        units = B * H
        min_rows = 256 if cap >= 4096 else 64
        for n in (ns, ntc):
            assert 1 <= n <= 128
            assert n == 1 or cap // n >= min_rows
        if wide == 2:
            assert G <= 4 and 2 <= ntc <= sms // units and cap // ntc >= 256
            assert units * ns <= 2 * sms
        elif wide:
            assert ntc == ns and units * ns <= (1 if G > 4 else 2) * sms
        else:
            assert units * ntc <= 2 * (2 if G > 4 else 4) * sms or ntc == 1   # never a third wave
            assert units * ns > (1 if G > 4 else 2) * sms                    # did not fit one wide wave


def test_decode_plan_argument_checks(kvq):
    assert kvq.lib.kvq_decode_plan_query(None, 8, SMS, None, None, None) == 1
    with pytest.raises(kvq.KvqError):
        _plan(kvq, 6, batch=1, n_kv_heads=4, capacity=100)          # 6 query heads over 4 kv heads
    with pytest.raises(kvq.KvqError):
        _plan(kvq, 8, sms=0, batch=1, n_kv_heads=4, capacity=100)
    with pytest.raises(kvq.KvqError):
        _plan(kvq, 8, batch=1, n_kv_heads=4, capacity=100, head_dim=96)


def test_layer_step_argument_checks(kvq):
    # checked on the host before any cache is touched: a layer count below 1,
    # missing per-layer arrays, unknown flags, and two layers on one cache
    lib = kvq.lib
    INVALID_ARG = 1   # KVQ_ERR_INVALID_ARG
    V = ctypes.c_void_p
    arr = lambda *xs: (V * len(xs))(*xs)
    one = arr(V(0x1000))
    st = lib.kvq_append_decode_layers(0, one, one, one, 1, one, one, 3, 1, 0.0, None, None, 0, None)
    assert st == INVALID_ARG and b"n_layers" in lib.kvq_last_error()
    st = lib.kvq_append_decode_layers(1, None, one, one, 1, one, one, 3, 1, 0.0, None, None, 0, None)
    assert st == INVALID_ARG and b"null per-layer array" in lib.kvq_last_error()
    st = lib.kvq_append_decode_layers(1, one, one, one, 1, one, one, 3, 1, 0.0, None, None, 4, None)
    assert st == INVALID_ARG and b"flags" in lib.kvq_last_error()
    # the same handle twice (never dereferenced: the check runs first)
    two = arr(V(0x1000), V(0x1000))
    st = lib.kvq_append_decode_layers(2, two, two, two, 1, two, two, 3, 1, 0.0, None, None, 0, None)
    assert st == INVALID_ARG and b"share one cache" in lib.kvq_last_error()
    assert lib.kvq_last_launch_count() == 0
