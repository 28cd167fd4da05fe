"""Helpers for the GPU tests: device models from the seeded recipe and raw-pointer views."""
import numpy as np
import torch

from synth import model as sm
from quantized_decode_gb300.kvfill import kv_pool_views, raw_view, write_kv  # noqa: F401


def to_dev(a):
    a = np.ascontiguousarray(a)
    return torch.from_numpy(a.view(np.uint8).reshape(-1).copy()).cuda()


def device_model(cfg, seed):
    from quantized_decode_gb300 import DeviceModel
    return DeviceModel(cfg, *sm.recipe(cfg, seed))


def fill_kv(engine, cfg, seed, T, page_perm=None):
    """Write seeded N(0,1) bf16 K/V for positions 0..T-1 of every layer through the page
    table (optionally shuffled first); returns the contiguous arrays [L][T][Hkv][d]."""
    ks, vs = [], []

    def draw(l):
        k, v = sm.kv_fill(cfg, seed, l, T)
        ks.append(k)
        vs.append(v)
        return k, v

    write_kv(engine, cfg, draw, T, page_perm)
    return ks, vs
