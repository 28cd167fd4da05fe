"""Helpers for the GPU tests: device models from the seeded recipe and raw-pointer views."""
import numpy as np
import torch

from synth import model as sm


class _RawCuda:
    def __init__(self, ptr, nbytes):
        self.__cuda_array_interface__ = {"shape": (nbytes,), "typestr": "|u1",
                                         "data": (int(ptr), False), "version": 3}


def raw_view(ptr, nbytes):
    """uint8 torch view of device memory owned by the engine (no copy)."""
    return torch.as_tensor(_RawCuda(ptr, nbytes), device="cuda")


def to_dev(a):
    a = np.ascontiguousarray(a)
    return torch.from_numpy(a.view(np.uint8).reshape(-1).copy()).cuda()


def device_model(cfg, seed):
    from quantized_decode_gb300 import DeviceModel
    return DeviceModel(cfg, *sm.recipe(cfg, seed))


def kv_pool_views(engine, cfg):
    """(k_pool, v_pool, page_table) torch views: pools as int16 [L][pages][Hkv][16][d]."""
    k, v, pt, n_pages = engine.debug_kv()
    shape = (cfg.n_layers, n_pages, cfg.n_kv_heads, 16, cfg.head_dim)
    nbytes = int(np.prod(shape)) * 2
    kp = raw_view(k, nbytes).view(torch.int16).view(shape)
    vp = raw_view(v, nbytes).view(torch.int16).view(shape)
    ptv = raw_view(pt, n_pages * 4).view(torch.int32)
    return kp, vp, ptv


def fill_kv(engine, cfg, seed, T, page_perm=None):
    """Write seeded N(0,1) bf16 K/V for positions 0..T-1 of every layer through the page
    table (optionally shuffled first); returns the contiguous arrays [L][T][Hkv][d]."""
    kp, vp, ptv = kv_pool_views(engine, cfg)
    n_pages = ptv.numel()
    if page_perm is not None:
        ptv.copy_(torch.from_numpy(np.ascontiguousarray(page_perm, dtype=np.int32)).cuda())
    table = ptv.cpu().numpy()
    ks, vs = [], []
    n_pg = (T + 15) // 16
    for l in range(cfg.n_layers):
        k, v = sm.kv_fill(cfg, seed, l, T)
        ks.append(k)
        vs.append(v)
        kpad = np.zeros((n_pg * 16, cfg.n_kv_heads, cfg.head_dim), np.uint16)
        vpad = np.zeros_like(kpad)
        kpad[:T], vpad[:T] = k, v
        # [pages][16][Hkv][d] -> [pages][Hkv][16][d]
        kb = torch.from_numpy(kpad.reshape(n_pg, 16, cfg.n_kv_heads, cfg.head_dim)
                              .transpose(0, 2, 1, 3).copy().view(np.int16)).cuda()
        vb = torch.from_numpy(vpad.reshape(n_pg, 16, cfg.n_kv_heads, cfg.head_dim)
                              .transpose(0, 2, 1, 3).copy().view(np.int16)).cuda()
        idx = torch.from_numpy(table[:n_pg].astype(np.int64)).cuda()
        kp[l].index_copy_(0, idx, kb)
        vp[l].index_copy_(0, idx, vb)
    torch.cuda.synchronize()
    engine.debug_kv(set_len=T)
    return ks, vs
