"""Write given K/V rows into an engine's paged cache through llm_debug_kv.

Used where a workload starts from a long cache without running its prefill (the
long-context and KV-length measurements, and the tests that check them): the values are
the caller's; this module only places them at the engine's layout, K and V pools
[L][pages][Hkv][16][d] bf16 behind one page table (logical page -> physical page).
"""
import numpy as np


class _RawCuda:
    def __init__(self, ptr, nbytes):
        self.__cuda_array_interface__ = {"shape": (nbytes,), "typestr": "|u1",
                                         "data": (int(ptr), False), "version": 3}


def raw_view(ptr, nbytes):
    """uint8 torch view of device memory owned by the engine (no copy)."""
    import torch
    return torch.as_tensor(_RawCuda(ptr, nbytes), device="cuda")


def kv_pool_views(engine, cfg):
    """(k_pool, v_pool, page_table) torch views: pools as int16 [L][pages][Hkv][16][d]."""
    import torch
    k, v, pt, n_pages = engine.debug_kv()
    shape = (cfg.n_layers, n_pages, cfg.n_kv_heads, 16, cfg.head_dim)
    nbytes = int(np.prod(shape)) * 2
    kp = raw_view(k, nbytes).view(torch.int16).view(shape)
    vp = raw_view(v, nbytes).view(torch.int16).view(shape)
    ptv = raw_view(pt, n_pages * 4).view(torch.int32)
    return kp, vp, ptv


def write_kv(engine, cfg, kv_of_layer, T, page_perm=None):
    """For every layer l, write kv_of_layer(l) -> (K, V) bf16 bits [T][Hkv][d] at positions
    0..T-1 through the page table (first replaced by page_perm when given), then set the
    sequence length to T.  Returns the page table in use (numpy int32)."""
    import torch
    kp, vp, ptv = kv_pool_views(engine, cfg)
    if page_perm is not None:
        ptv.copy_(torch.from_numpy(np.ascontiguousarray(page_perm, dtype=np.int32)).cuda())
    table = ptv.cpu().numpy()
    n_pg = (T + 15) // 16
    idx = torch.from_numpy(table[:n_pg].astype(np.int64)).cuda()
    for l in range(cfg.n_layers):
        k, v = kv_of_layer(l)
        for src, pool in ((k, kp), (v, vp)):
            pad = np.zeros((n_pg * 16, cfg.n_kv_heads, cfg.head_dim), np.uint16)
            pad[:T] = src
            # [pages][16][Hkv][d] -> [pages][Hkv][16][d]
            blk = torch.from_numpy(pad.reshape(n_pg, 16, cfg.n_kv_heads, cfg.head_dim)
                                   .transpose(0, 2, 1, 3).copy().view(np.int16)).cuda()
            pool[l].index_copy_(0, idx, blk)
    torch.cuda.synchronize()
    engine.debug_kv(set_len=T)
    return table
