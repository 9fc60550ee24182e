"""Drive a cache through the public calls: prefill a workload's starting state
and run one speculative round.  Every step is a libqs call; this module only
sequences them and moves synthetic inputs to the device.
"""
import numpy as np

from . import qs, synthetic


def prefill(cache, w, stream=None, max_groups=None):
    """Bring ``cache`` to the workload's starting state through the public
    calls: for each group, append G tokens, commit them (rollback of 0, or of
    G for sequences that already hold all their groups), flush the sequences
    that still need groups; then append the buffer tokens and commit each
    sequence's fill level.  Quantization happens on the device."""
    import torch
    dev = cache.state.device
    B, H, G = w.B, w.H, w.G
    ng = np.array(w.n_groups if max_groups is None else [min(n, max_groups) for n in w.n_groups])
    fill = np.array(w.fill)
    qs.qs_state_reset(cache, stream)
    for g in range(int(ng.max(initial=0))):
        k = np.empty((B, H, G, w.D), np.float16)
        v = np.empty_like(k)
        for b in range(B):
            if g < ng[b]:
                k[b], v[b] = synthetic.kv_chunk(w, b, g)
            else:
                k[b] = 0
                v[b] = 0
        kd = torch.from_numpy(k).to(dev)
        vd = torch.from_numpy(v).to(dev)
        qs.qs_buffer_append(cache, kd, vd, stream)
        drop = torch.from_numpy(np.where(g < ng, 0, G).astype(np.int32)).to(dev)
        qs.qs_buffer_rollback(cache, drop, stream)
        mask = torch.from_numpy((g < ng).astype(np.uint8)).to(dev)
        qs.qs_quantize_flush(cache, mask, stream)
    fmax = int(fill.max(initial=0))
    if fmax:
        k = np.zeros((B, H, fmax, w.D), np.float16)
        v = np.zeros_like(k)
        for b in range(B):
            if fill[b]:
                k[b, :, :fill[b]], v[b, :, :fill[b]] = synthetic.kv_tokens(w, b, int(ng[b]) * G,
                                                                          int(fill[b]))
        qs.qs_buffer_append(cache, torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev), stream)
        drop = torch.from_numpy((fmax - fill).astype(np.int32)).to(dev)
        qs.qs_buffer_rollback(cache, drop, stream)
    return ng, fill
