"""A small Python front end over the C ABI: PyTorch allocates the device and page-locked host
memory and supplies the CUDA stream; every step of the hot path runs in libverkv's kernels.

    eng = VerKV(shape)                   # workspace + context on the current CUDA device/stream
    eng.load(tau, kv)                    # numpy -> device tensors and a page-locked host copy
    eng.compress(eta, n_sink, n_local, seed)   # verkv_poissoncomp + verkv_sketch_build
    eng.attend(layer, q_dev, eps, delta)        # verkv_attend_verified
    o, lse, stats = eng.fetch_refine()          # verkv_fetch_refine
"""
import numpy as np
import torch

from . import binding as B


def _check_dense(t, shape, dev, name):
    """The library reads tensors as dense row-major arrays: refuse anything else."""
    if t.device != dev or not t.is_contiguous() or t.numel() != int(np.prod(shape)):
        raise ValueError(f"{name}: a contiguous {list(shape)} tensor on {dev} is required")


def default_cap(n, eta):
    """Pivotal capacity: eta n plus 8 standard deviations of a Poisson sample size, plus 64,
    rounded up to a multiple of 16 (so that every pivotal item's id and r lists start on 16-byte
    boundaries and can be bulk-copied), at most n."""
    m = eta * n
    c = int(np.ceil(m + 8.0 * np.sqrt(m)) + 64)
    return int(min(n, (c + 15) // 16 * 16))


class VerKV:
    def __init__(self, batch, layers, kv_heads, q_per_kv, head_dim, n, cap, device=None,
                 fetch_mode=B.VERKV_FETCH_ZEROCOPY, sketch_format=B.VERKV_SKETCH_EXACT, seq0=0):
        """seq0: the index of this context's first sequence in a batch split over several
        contexts (its Poisson draws are then those of that sequence; see
        verkv_set_sequence_offset)."""
        self.dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
        self.shape = B.verkv_shape(batch, layers, kv_heads, q_per_kv, head_dim, n, cap)
        self.B, self.L, self.h, self.G, self.d, self.n, self.cap = (
            batch, layers, kv_heads, q_per_kv, head_dim, n, cap)
        self.units = batch * layers * kv_heads
        self.sketch_format = sketch_format
        self.W = (n + 31) // 32
        ws = B.verkv_workspace_size(self.shape)
        if ws == 0:
            raise B.VerkvError(B.VERKV_EINVAL, "invalid shape")
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=self.dev)
        self.stream = torch.cuda.current_stream(self.dev)
        self.ctx = B.verkv_create(self.dev.index, self.stream.cuda_stream, self.shape,
                                  self.workspace.data_ptr(), ws)
        if fetch_mode != B.VERKV_FETCH_ZEROCOPY:
            B.verkv_set_fetch_mode(self.ctx, fetch_mode)
        if seq0:
            B.verkv_set_sequence_offset(self.ctx, seq0)
        dv = self.dev
        u, hq = self.units, batch * kv_heads * q_per_kv
        self.r_full = torch.empty((u, n), dtype=torch.float32, device=dv)
        self.p_ids = torch.empty((u, cap), dtype=torch.int32, device=dv)
        self.p_r = torch.empty((u, cap), dtype=torch.float32, device=dv)
        self.p_kv = torch.empty((u, cap, 2, head_dim), dtype=torch.int16, device=dv)
        self.p_count = torch.empty((u,), dtype=torch.int32, device=dv)
        self.p_res = torch.empty((u, self.W), dtype=torch.int32, device=dv)
        self.p_c = torch.empty((u,), dtype=torch.float32, device=dv)
        self.pivotal = B.verkv_pivotal(self.p_ids.data_ptr(), self.p_r.data_ptr(),
                                       self.p_kv.data_ptr(), self.p_count.data_ptr(),
                                       self.p_res.data_ptr(), self.p_c.data_ptr())
        self.o = torch.empty((hq, head_dim), dtype=torch.float32, device=dv)
        self.lse = torch.empty((hq,), dtype=torch.float32, device=dv)
        self.stats = torch.empty((hq, 16), dtype=torch.int32, device=dv)  # verkv_head_stats
        self.fetch_ids = torch.empty((batch * kv_heads, n), dtype=torch.int32, device=dv)
        self.fetch_counts = torch.empty((batch * kv_heads,), dtype=torch.int32, device=dv)
        self.tau = self.kv = self.sketch = self.host_kv = None

    # --------------------------------------------------------------------------------------------
    def load(self, tau, kv):
        """tau float32 [units][n], kv uint16 (bf16 bits) [units][n][2][d] (numpy or torch CPU)."""
        tau_t = torch.as_tensor(np.ascontiguousarray(tau, dtype=np.float32)).reshape(self.units, self.n)
        kv_t = torch.as_tensor(np.ascontiguousarray(kv).view(np.int16)).reshape(
            self.units, self.n, 2, self.d)
        self.tau = tau_t.to(self.dev)
        self.host_kv = torch.empty(kv_t.shape, dtype=torch.int16, pin_memory=True)
        self.host_kv.copy_(kv_t)
        self.kv = self.host_kv.to(self.dev)
        if self.sketch_format == B.VERKV_SKETCH_EXACT:
            self.sketch = torch.empty((self.units, self.n, self.d), dtype=torch.int16, device=self.dev)
        else:
            nbytes = B.verkv_sketch_bytes(self.shape, self.sketch_format)
            self.sketch = torch.empty((self.units, self.n, nbytes // (self.units * self.n)),
                                      dtype=torch.uint8, device=self.dev)
        self.sketch_desc = B.verkv_sketch(self.sketch_format, self.sketch.data_ptr())

    def load_device(self, tau, kv, host_kv):
        """Adopt tensors that already exist: tau float32 [units][n] and kv int16 (bf16 bits)
        [units][n][2][d] on this device, host_kv the same layout in page-locked host memory."""
        _check_dense(tau, (self.units, self.n), self.dev, "tau")
        _check_dense(kv, (self.units, self.n, 2, self.d), self.dev, "kv")
        if not (host_kv.is_pinned() and host_kv.is_contiguous() and host_kv.numel() == kv.numel()):
            raise ValueError("host_kv: a contiguous page-locked copy of kv is required")
        self.tau = tau.reshape(self.units, self.n)
        self.kv = kv.reshape(self.units, self.n, 2, self.d)
        self.host_kv = host_kv.reshape(self.units, self.n, 2, self.d)
        if self.sketch_format == B.VERKV_SKETCH_EXACT:
            self.sketch = torch.empty((self.units, self.n, self.d), dtype=torch.int16, device=self.dev)
        else:
            nbytes = B.verkv_sketch_bytes(self.shape, self.sketch_format)
            self.sketch = torch.empty((self.units, self.n, nbytes // (self.units * self.n)),
                                      dtype=torch.uint8, device=self.dev)
        self.sketch_desc = B.verkv_sketch(self.sketch_format, self.sketch.data_ptr())

    def compress(self, eta, n_sink, n_local, seed):
        B.verkv_poissoncomp(self.ctx, self.tau.data_ptr(), eta, B.verkv_hset(n_sink, n_local),
                            seed, self.kv.data_ptr(), self.r_full.data_ptr(), self.pivotal)
        B.verkv_sketch_build(self.ctx, self.kv.data_ptr(), self.sketch_format,
                             self.sketch.data_ptr())

    def attend(self, layer, q, eps, delta, with_ids=True):
        """q: device bf16 (int16 view) [batch][kv_heads * q_per_kv][d], contiguous."""
        _check_dense(q, (self.B, self.h * self.G, self.d), self.dev, "q")
        self._q = q
        ids = self.fetch_ids.data_ptr() if with_ids else None
        cnt = self.fetch_counts.data_ptr() if with_ids else None
        B.verkv_attend_verified(self.ctx, layer, q.data_ptr(), self.pivotal,
                                self.r_full.data_ptr(), self.sketch_desc, eps, delta, ids, cnt)
        self._ids, self._cnt = ids, cnt

    def fetch_refine(self, o=None, lse=None, stats=None):
        o = self.o if o is None else o
        lse = self.lse if lse is None else lse
        stats = self.stats if stats is None else stats
        B.verkv_fetch_refine(self.ctx, self._ids, self._cnt, self.host_kv.data_ptr(),
                             o.data_ptr(), lse.data_ptr() if lse is not None else None,
                             stats.data_ptr() if stats is not None else None)
        return o, lse, stats

    def attend_dense_host(self, layer, q, o=None, lse=None):
        """The offloaded-dense baseline: exact attention with every row read from the host."""
        o = torch.empty_like(self.o) if o is None else o
        lse = torch.empty_like(self.lse) if lse is None else lse
        B.verkv_attend_dense_host(self.ctx, layer, q.data_ptr(), self.host_kv.data_ptr(),
                                  o.data_ptr(), lse.data_ptr())
        return o, lse

    def set_shortlist(self, size):
        """Shortlist variant: at most `size` tokens per KV head may be fetched (0: off)."""
        B.verkv_set_shortlist(self.ctx, size)

    def shortlist_bitmap(self):
        out = torch.empty((self.B * self.h, self.W), dtype=torch.int32, device=self.dev)
        B.verkv_shortlist_bitmap(self.ctx, out.data_ptr())
        return out

    def selection_bitmap(self):
        out = torch.empty((self.B * self.h * self.G, self.W), dtype=torch.int32, device=self.dev)
        B.verkv_selection_bitmap(self.ctx, out.data_ptr())
        return out

    def sync(self):
        B.verkv_sync(self.ctx)

    def close(self):
        if self.ctx is not None:
            B.verkv_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001 -- interpreter shutdown
            pass


def stats_to_dict(stats):
    """[hq][16] int32 tensor of verkv_head_stats -> dict of numpy arrays."""
    a = stats.cpu().numpy()
    f = a[:, :10].view(np.float32)
    out = {k: f[:, i].copy() for i, k in enumerate(B.STATS_FLOAT_FIELDS)}
    for i, k in enumerate(B.STATS_INT_FIELDS):
        out[k] = a[:, 10 + i].copy()
    return out
