"""The paged-attention input generator: the torch path that builds the
device pool gives the numpy path's bits (torch on the CPU here), so the
GPU tests and the bench draw exactly the oracle's inputs."""
import numpy as np
import torch

import synth


def test_paged_attention_torch_equals_numpy():
    p = synth.PagedAttention("t", (37, 100, 64), 3, 8, 2, 128, 16, 21, shared_prefix=32)
    d = synth.gen_paged_attention(p)
    t = synth.gen_paged_attention_torch(p, torch.device("cpu"), chunk=5000)
    for k in ("kc", "vc"):
        assert t[k].dtype == torch.int8 and (t[k].numpy() == d[k]).all(), k
    for k in ("kd", "vd", "q"):
        assert (t[k].numpy().view(np.uint16) == d[k]).all(), k
    for k in ("page_table", "seq_len", "row_seq", "row_pos"):
        assert (t[k].numpy() == d[k]).all(), k
