"""On-disk container for quantized layers: a safetensors file plus
quantize_config.json.

The GPTQ practical guide (m.lqnn.cn/news/117696, §3.4) says a quantized model
is saved as a directory holding safetensors weight files and a
quantize_config.json, and that every loader reads that config to learn the
bit width, the group size and whether desc_act was used (§3.4, §5.2); §3.3
names the knobs bits, group_size, desc_act and damp_percent.  The pages fix
nothing else, so:

  * tensors, per layer `name`: `name.qweight` (int32 [d_col*bits/32, d_row]),
    `name.qzeros` (int32 [G, d_row*bits/32]), `name.scales` (fp32 [G, d_row])
    and `name.g_idx` (int32 [d_col]), in the layouts of gptq_pack;
  * quantize_config.json: bits, group_size, desc_act, damp_percent and sym
    (the ms-swift page's GptqConfig example names sym), plus the packing
    layout under "pack_layout";
  * the safetensors file follows the format's public layout: an 8-byte
    little-endian header length, a JSON header (padded with spaces to a
    multiple of 8 bytes) mapping each tensor name to its dtype, shape and
    [begin, end) byte range in the data section, an optional "__metadata__"
    map of strings, then the data section with the tensors back to back in
    little-endian order, covering it with no gap.

Host-side file I/O only; nothing here runs on the GPU.
"""
from __future__ import annotations

import json
import os
import struct

import numpy as np

from .workloads import QuantConfig

_DTYPES = {
    np.dtype("int32"): "I32",
    np.dtype("int64"): "I64",
    np.dtype("uint8"): "U8",
    np.dtype("int8"): "I8",
    np.dtype("float16"): "F16",
    np.dtype("float32"): "F32",
    np.dtype("float64"): "F64",
}
_NP = {v: k for k, v in _DTYPES.items()}

CONFIG_NAME = "quantize_config.json"
WEIGHTS_NAME = "model.safetensors"
PACK_LAYOUT = ("qweight int32 [d_col*bits/32, d_row]: column r is row r's codes as one LSB-first "
               "bit stream along the input dimension; qzeros int32 [G, d_row*bits/32]: LSB-first "
               "along rows, stored without offset; scales fp32 [G, d_row]; g_idx int32 [d_col]")


def _host(a) -> np.ndarray:
    """numpy view of a host array or a (device) torch tensor."""
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a)


def write_safetensors(path: str, tensors: dict, metadata: dict | None = None) -> None:
    """Write `tensors` (name -> array) to `path`; names are stored sorted."""
    header: dict = {}
    blobs = []
    offset = 0
    for name in sorted(tensors):
        a = _host(tensors[name])
        if a.dtype not in _DTYPES:
            raise ValueError(f"{name}: unsupported dtype {a.dtype}")
        raw = a.astype(a.dtype.newbyteorder("<"), copy=False).tobytes()
        header[name] = {"dtype": _DTYPES[a.dtype], "shape": list(a.shape),
                        "data_offsets": [offset, offset + len(raw)]}
        blobs.append(raw)
        offset += len(raw)
    if metadata:
        header["__metadata__"] = {str(k): str(v) for k, v in metadata.items()}
    hb = json.dumps(header, separators=(",", ":")).encode("utf-8")
    hb += b" " * ((-len(hb)) % 8)
    tmp = path + ".tmp"
    with open(tmp, "wb") as f:
        f.write(struct.pack("<Q", len(hb)))
        f.write(hb)
        for raw in blobs:
            f.write(raw)
    os.replace(tmp, path)


def read_safetensors(path: str) -> tuple[dict, dict]:
    """(name -> array, metadata).  Raises ValueError on a malformed file."""
    with open(path, "rb") as f:
        buf = f.read()
    if len(buf) < 8:
        raise ValueError("file shorter than the header length field")
    (n,) = struct.unpack("<Q", buf[:8])
    if 8 + n > len(buf):
        raise ValueError("header runs past the end of the file")
    header = json.loads(buf[8:8 + n].decode("utf-8"))
    data = memoryview(buf)[8 + n:]
    metadata = header.pop("__metadata__", {}) or {}
    spans = []
    out = {}
    for name, d in header.items():
        if d["dtype"] not in _NP:
            raise ValueError(f"{name}: unsupported dtype {d['dtype']}")
        dt = _NP[d["dtype"]].newbyteorder("<")
        b, e = (int(x) for x in d["data_offsets"])
        shape = tuple(int(s) for s in d["shape"])
        if not (0 <= b <= e <= len(data)):
            raise ValueError(f"{name}: byte range [{b}, {e}) outside the data section")
        if int(np.prod(shape, dtype=np.int64)) * dt.itemsize != e - b:
            raise ValueError(f"{name}: byte range does not match dtype and shape")
        spans.append((b, e, name))
        out[name] = np.frombuffer(data[b:e], dtype=dt).reshape(shape).astype(dt.newbyteorder("="))
    spans.sort()
    for (b0, e0, n0), (b1, e1, n1) in zip(spans, spans[1:]):
        if b1 < e0:
            raise ValueError(f"{n0} and {n1} overlap")
        if b1 > e0:
            raise ValueError(f"unused bytes between {n0} and {n1}")
    if spans and (spans[0][0] != 0 or spans[-1][1] != len(data)):
        raise ValueError("the tensors do not cover the data section exactly")
    return out, metadata


def config_dict(cfg: QuantConfig) -> dict:
    return {"bits": int(cfg.bits), "group_size": int(cfg.group_size), "desc_act": bool(cfg.desc_act),
            "damp_percent": float(cfg.damp_percent), "sym": bool(cfg.sym), "pack_layout": PACK_LAYOUT}


def save_quantized(directory: str, layers: dict, cfg: QuantConfig) -> None:
    """Write `layers` (name -> mapping or object with qweight, qzeros,
    scales, g_idx) and the config into `directory`."""
    os.makedirs(directory, exist_ok=True)
    tensors = {}
    for name, layer in layers.items():
        get = layer.get if isinstance(layer, dict) else (lambda k, _l=layer: getattr(_l, k))
        qweight, qzeros = _host(get("qweight")), _host(get("qzeros"))
        scales, g_idx = _host(get("scales")), _host(get("g_idx"))
        d_row = qweight.shape[1]
        d_col = qweight.shape[0] * 32 // cfg.bits
        G = 1 if cfg.group_size == -1 else d_col // cfg.group_size
        if qweight.dtype != np.int32 or qzeros.dtype != np.int32 or g_idx.dtype != np.int32:
            raise ValueError(f"{name}: qweight, qzeros and g_idx must be int32")
        if qzeros.shape != (G, d_row * cfg.bits // 32) or scales.shape != (G, d_row) or g_idx.shape != (d_col,):
            raise ValueError(f"{name}: shapes do not match bits={cfg.bits}, group_size={cfg.group_size}")
        tensors[f"{name}.qweight"] = qweight
        tensors[f"{name}.qzeros"] = qzeros
        tensors[f"{name}.scales"] = scales.astype(np.float32, copy=False)
        tensors[f"{name}.g_idx"] = g_idx
    write_safetensors(os.path.join(directory, WEIGHTS_NAME), tensors,
                      metadata={"format": "gptq", "layers": ",".join(sorted(layers))})
    with open(os.path.join(directory, CONFIG_NAME), "w") as f:
        json.dump(config_dict(cfg), f, indent=2, sort_keys=True)
        f.write("\n")


def load_quantized(directory: str) -> tuple[dict, QuantConfig]:
    """(name -> {qweight, qzeros, scales, g_idx}, config) from `directory`."""
    with open(os.path.join(directory, CONFIG_NAME)) as f:
        c = json.load(f)
    cfg = QuantConfig(bits=int(c["bits"]), group_size=int(c["group_size"]), desc_act=bool(c["desc_act"]),
                      damp_percent=float(c["damp_percent"]), sym=bool(c.get("sym", False)))
    tensors, _meta = read_safetensors(os.path.join(directory, WEIGHTS_NAME))
    layers: dict = {}
    for key, a in tensors.items():
        name, _, part = key.rpartition(".")
        if part not in ("qweight", "qzeros", "scales", "g_idx") or not name:
            raise ValueError(f"unexpected tensor {key}")
        layers.setdefault(name, {})[part] = a
    for name, parts in layers.items():
        if len(parts) != 4:
            raise ValueError(f"{name}: incomplete layer ({sorted(parts)})")
    return layers, cfg
