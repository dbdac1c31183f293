"""Shared test plumbing: move a synth layer to the device and to the oracle."""
import numpy as np

import oracle
import synth


def to_oracle(layer) -> "oracle.Tensor":
    return oracle.Tensor(layer["fmt"], layer["N"], layer["K"], layer["w"], layer["scales"],
                         layer["zeros"], layer["g_idx"], layer["group"], layer["scale2"])


def to_device(layer):
    import torch

    def dev(a):
        if a is None:
            return None
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return torch.from_numpy(a).cuda()
    return {k: dev(layer[k]) for k in ("w", "scales", "zeros", "g_idx")}


def x_device(bits_or_f32):
    import torch
    a = np.ascontiguousarray(bits_or_f32)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a.astype(np.float32)).cuda()


def aux_for(layer, d, x_dtype=None, out_dtype=0):
    import bit_block_quantized_gb300 as q4
    return q4.make_aux(scale2=layer["scale2"], zeros=d["zeros"], g_idx=d["g_idx"],
                       group=layer["group"], x_dtype=x_dtype, out_dtype=out_dtype, fmt=layer["fmt"])


def within_tolerance(y_gpu, y_ref, bound):
    tol = oracle.gemv_tolerance(bound)
    err = np.abs(np.asarray(y_gpu, np.float64) - y_ref)
    return bool(np.all(err <= tol)), float(np.max(err / tol))


def oracle_gemv_all_rows(t, xf, threads=None):
    """oracle.gemv over every row, the rows split into chunks that run on
    host threads (the C oracle releases the GIL); the per-row arithmetic is
    the oracle's own, so the result is identical to one call."""
    import os
    from concurrent.futures import ThreadPoolExecutor

    threads = threads or min(16, os.cpu_count() or 1)
    chunks = np.array_split(np.arange(t.N), max(1, min(threads * 4, t.N)))
    with ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(lambda r: oracle.gemv(t, xf, rows=r), chunks))
    return (np.concatenate([p[0] for p in parts], axis=1), np.concatenate([p[1] for p in parts], axis=1))
