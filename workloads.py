"""Device-resident synthetic workloads, built through the library's public API.

Values come from the seeded generator (``synth``, identical on host and
device); weight preparation is the library's own: blockwise Walsh-Hadamard
rotation (PQ2_0 only, rotate then quantize) and the device quantizers.  Used
by the GPU tests and the benchmark; the oracle rebuilds any row of these
matrices on the host from the same seeds.
"""
import numpy as np
import torch

import quantized_weight_streaming_gb300 as kq
import synth


def _fmt_name(fmt):
    if isinstance(fmt, str):
        return fmt
    return {kq.KQ_Q8_0: "q8_0", kq.KQ_PQ2_0: "pq2_0", kq.KQ_SCALE4: "scale4"}[fmt]


def build_matrix(fmt, n, k, seed, stream, tmp=None, device="cuda", had_block=None, signs=None):
    """Quantized n x k matrix from generator stream (seed, stream).  tmp, if
    given, is a float32 device tensor with at least n*k elements used as the
    fp32 staging buffer.  PQ2_0 weights are rotated first (W' = W R^T): by
    H_128/sqrt(128), or with had_block=1024 and signs (an int8 device tensor
    of k entries, or None) by the page's H_1024 S / 32."""
    W = kq.QMatrix(fmt, n, k, device=device, had_block=had_block, signs=signs)
    if tmp is None or tmp.numel() < n * k:
        tmp = torch.empty(n * k, dtype=torch.float32, device=device)
    w = tmp[: n * k]
    synth.fill_device(w.data_ptr(), "w", n * k, seed, stream, cuda_stream=torch.cuda.current_stream().cuda_stream)
    if _fmt_name(fmt) == "pq2_0":
        kq.kq_rotate_blockwise(w, w, n, k, W.had_block, signs)
        kq.kq_quantize_pq2_0_device(W, w)
    elif _fmt_name(fmt) == "scale4":
        kq.kq_quantize_scale4_device(W, w)
    else:
        kq.kq_quantize_q8_0_device(W, w)
    return W


def build_signs(k, seed, stream, device="cuda"):
    """(host int8 array, device int8 tensor) of a seeded +-1 sign vector."""
    h = synth.sign_vector(k, seed, stream)
    return h, torch.from_numpy(h).to(device)


def build_activation(k, seed, stream, rows=1, device="cuda"):
    x = torch.empty(rows * k, dtype=torch.float32, device=device)
    synth.fill_device(x.data_ptr(), "x", rows * k, seed, stream, cuda_stream=torch.cuda.current_stream().cuda_stream)
    return x


class DecodeWorkload:
    """A decode-step workload: every projection quantized on the device, one
    activation vector per projection packed into x, outputs packed into y.

    linked=True builds the step with the model's dependencies instead
    (``synth.decode_links``): only the first projection reads a packed input,
    every later one reads its group's input or alpha times an earlier output,
    stage by stage, in one cooperative launch per step."""

    def __init__(self, config, seed=0, device="cuda", limit=None, linked=False, rotation=None):
        """rotation="page": PQ2_0 matrices use the page's rotation, 1024-point
        blocks with one seeded sign vector per K width (shared by every matrix
        of that width)."""
        self.config = config
        self.seed = seed
        self.linked = linked
        self.rotation = rotation
        self.mats_spec = synth.workload(config)
        if limit:
            self.mats_spec = self.mats_spec[:limit]
        self.links = synth.decode_links(config)[: len(self.mats_spec)] if linked else None
        big = max(n * k for _, _, n, k in self.mats_spec)
        tmp = torch.empty(big, dtype=torch.float32, device=device)
        self.mats = []
        self.signs = {}  # K width -> (host, device) signs of the page's rotation
        for i, (_, fmt, n, k) in enumerate(self.mats_spec):
            had, sd = None, None
            if rotation == "page" and fmt == synth.PQ2_0:
                if k not in self.signs:
                    self.signs[k] = build_signs(k, seed, synth.stream_id(config, synth.ROLE_S, k), device)
                had, sd = 1024, self.signs[k][1]
            self.mats.append(build_matrix(fmt, n, k, seed, synth.stream_id(config, synth.ROLE_W, i), tmp, device,
                                          had_block=had, signs=sd))
        del tmp
        # packed inputs: every projection's own (unlinked), or those of the
        # projections whose link is SRC_PACKED (linked), in list order
        packed = [i for i in range(len(self.mats_spec))
                  if not linked or self.links[i][0] == synth.SRC_PACKED]
        self.packed = packed
        self.x_offsets = np.cumsum([0] + [self.mats_spec[i][3] for i in packed])
        self.y_offsets = np.cumsum([0] + [n for _, _, n, _ in self.mats_spec])
        self.x = torch.empty(int(self.x_offsets[-1]), dtype=torch.float32, device=device)
        for slot, i in enumerate(packed):
            off, k = int(self.x_offsets[slot]), self.mats_spec[i][3]
            synth.fill_device(self.x[off:].data_ptr(), "x", k, seed, synth.stream_id(config, synth.ROLE_X, i),
                              cuda_stream=torch.cuda.current_stream().cuda_stream)
        self.y = torch.empty(int(self.y_offsets[-1]), dtype=torch.float32, device=device)
        self.plan = kq.DecodePlan(self.mats, self.links)
        assert self.plan.x_floats == self.x.numel() and self.plan.y_floats == self.y.numel()
        nb = self.plan.workspace_bytes
        self.ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=device) if nb else None

    @property
    def weight_bytes(self):
        return self.plan.weight_bytes

    @property
    def activation_bytes(self):
        """fp32 activations read (every projection's input, also when it is an
        earlier output) plus outputs written."""
        return 4 * sum(n + k for _, _, n, k in self.mats_spec)

    def step(self, stream=None):
        self.plan.step(self.x, self.y, self.ws, stream=stream)

    def host_rows(self, i, rows):
        """(W rows fp32, x fp32) of projection i regenerated on the host."""
        _, _, n, k = self.mats_spec[i]
        w = synth.matrix_rows_host(n, k, rows, self.seed, synth.stream_id(self.config, synth.ROLE_W, i))
        x = synth.fill_host("x", k, self.seed, synth.stream_id(self.config, synth.ROLE_X, i))
        return w, x

    def close(self):
        self.plan.close()
