"""The on-disk container: safetensors byte layout checked against bytes built
by hand, round trips, malformed files, and quantize_config.json."""
import json
import os
import struct

import numpy as np
import pytest

import oracle as O
from post_weight_quantization_31_b300 import container as C
from post_weight_quantization_31_b300 import workloads as wl


def test_reads_a_hand_built_file(tmp_path):
    # two tensors, header written by hand, data little-endian back to back
    header = {"a": {"dtype": "I32", "shape": [2], "data_offsets": [0, 8]},
              "b": {"dtype": "F32", "shape": [1, 2], "data_offsets": [8, 16]},
              "__metadata__": {"k": "v"}}
    hb = json.dumps(header).encode()
    data = struct.pack("<ii", 7, -3) + struct.pack("<ff", 1.5, -0.25)
    p = tmp_path / "h.safetensors"
    p.write_bytes(struct.pack("<Q", len(hb)) + hb + data)
    t, meta = C.read_safetensors(str(p))
    assert meta == {"k": "v"}
    assert t["a"].dtype == np.int32 and t["a"].tolist() == [7, -3]
    assert t["b"].shape == (1, 2) and t["b"].tolist() == [[1.5, -0.25]]


def test_writer_layout(tmp_path):
    p = str(tmp_path / "w.safetensors")
    C.write_safetensors(p, {"z": np.arange(3, dtype=np.int32), "a": np.ones((2, 2), np.float16)},
                        metadata={"format": "gptq"})
    raw = open(p, "rb").read()
    (n,) = struct.unpack("<Q", raw[:8])
    assert n % 8 == 0                                   # header padded to 8 bytes
    header = json.loads(raw[8:8 + n])
    assert header["__metadata__"] == {"format": "gptq"}
    assert header["a"] == {"dtype": "F16", "shape": [2, 2], "data_offsets": [0, 8]}
    assert header["z"] == {"dtype": "I32", "shape": [3], "data_offsets": [8, 20]}
    assert raw[8 + n:8 + n + 8] == np.ones(4, np.float16).tobytes()
    assert raw[8 + n + 8:] == struct.pack("<iii", 0, 1, 2)


@pytest.mark.parametrize("dt", ["int32", "int64", "uint8", "int8", "float16", "float32", "float64"])
def test_round_trip_every_dtype(tmp_path, dt):
    rng = np.random.Generator(np.random.PCG64(3))
    a = (rng.standard_normal((5, 7)) * 50).astype(dt)
    p = str(tmp_path / "r.safetensors")
    C.write_safetensors(p, {"x": a, "empty": np.zeros((0, 3), dt)})
    t, _ = C.read_safetensors(p)
    assert np.array_equal(t["x"], a) and t["x"].dtype == a.dtype
    assert t["empty"].shape == (0, 3)


def _corrupt(tmp_path, header, data=b"\0" * 16):
    hb = json.dumps(header).encode()
    p = tmp_path / "bad.safetensors"
    p.write_bytes(struct.pack("<Q", len(hb)) + hb + data)
    return str(p)


def test_rejects_malformed_files(tmp_path):
    with pytest.raises(ValueError):      # range past the data
        C.read_safetensors(_corrupt(tmp_path, {"a": {"dtype": "I32", "shape": [8], "data_offsets": [0, 32]}}))
    with pytest.raises(ValueError):      # size does not match the shape
        C.read_safetensors(_corrupt(tmp_path, {"a": {"dtype": "I32", "shape": [3], "data_offsets": [0, 8]}}))
    with pytest.raises(ValueError):      # overlapping tensors
        C.read_safetensors(_corrupt(tmp_path, {"a": {"dtype": "I32", "shape": [2], "data_offsets": [0, 8]},
                                               "b": {"dtype": "I32", "shape": [2], "data_offsets": [4, 12]}}))
    with pytest.raises(ValueError):      # a gap between tensors
        C.read_safetensors(_corrupt(tmp_path, {"a": {"dtype": "I32", "shape": [1], "data_offsets": [0, 4]},
                                               "b": {"dtype": "I32", "shape": [2], "data_offsets": [8, 16]}}))
    with pytest.raises(ValueError):      # trailing bytes not covered by any tensor
        C.read_safetensors(_corrupt(tmp_path, {"a": {"dtype": "I32", "shape": [2], "data_offsets": [0, 8]}}))
    p = tmp_path / "short.safetensors"
    p.write_bytes(struct.pack("<Q", 100) + b"{}")
    with pytest.raises(ValueError):      # header longer than the file
        C.read_safetensors(str(p))


def _packed_layer(d_row, d_col, cfg, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    codes = rng.integers(0, 1 << cfg.bits, size=(d_row, d_col))
    G = 1 if cfg.group_size == -1 else d_col // cfg.group_size
    zeros = rng.integers(0, 1 << cfg.bits, size=(G, d_row))
    perm = rng.permutation(d_col) if cfg.desc_act else np.arange(d_col)
    return {"qweight": O.pack_qweight(codes, cfg.bits), "qzeros": O.pack_qzeros(zeros, cfg.bits),
            "scales": rng.uniform(1e-3, 1e-2, size=(G, d_row)).astype(np.float32),
            "g_idx": O.group_index(perm, cfg.group_size).astype(np.int32)}, codes, zeros


def test_save_and_load_quantized(tmp_path):
    cfg = wl.QuantConfig(bits=3, group_size=64, desc_act=True, damp_percent=0.02, sym=True)
    l0, codes, zeros = _packed_layer(64, 256, cfg, 1)
    l1, _, _ = _packed_layer(32, 128, cfg, 2)
    C.save_quantized(str(tmp_path), {"model.layers.0.self_attn.q_proj": l0, "mlp.down": l1}, cfg)
    conf = json.load(open(os.path.join(tmp_path, C.CONFIG_NAME)))
    assert {k: conf[k] for k in ("bits", "group_size", "desc_act", "damp_percent", "sym")} == \
        {"bits": 3, "group_size": 64, "desc_act": True, "damp_percent": 0.02, "sym": True}
    layers, cfg2 = C.load_quantized(str(tmp_path))
    assert cfg2 == cfg
    assert sorted(layers) == ["mlp.down", "model.layers.0.self_attn.q_proj"]
    got = layers["model.layers.0.self_attn.q_proj"]
    for k in ("qweight", "qzeros", "scales", "g_idx"):
        assert np.array_equal(got[k], l0[k]) and got[k].dtype == l0[k].dtype
    # the reloaded layer decodes to the same weights
    assert np.array_equal(O.unpack_qweight(got["qweight"], 3, 256), codes)
    assert np.array_equal(O.unpack_qzeros(got["qzeros"], 3, 64), zeros)


def test_save_rejects_inconsistent_layers(tmp_path):
    cfg = wl.QuantConfig(bits=4, group_size=128)
    layer, _, _ = _packed_layer(32, 256, cfg, 3)
    bad = dict(layer, scales=layer["scales"][:1])
    with pytest.raises(ValueError):
        C.save_quantized(str(tmp_path), {"x": bad}, cfg)
    bad = dict(layer, qweight=layer["qweight"].astype(np.int64))
    with pytest.raises(ValueError):
        C.save_quantized(str(tmp_path), {"x": bad}, cfg)
