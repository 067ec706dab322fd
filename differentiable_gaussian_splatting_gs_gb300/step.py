"""One training step of one or more views through the five entry points.

Per view (the phases preprocessing, rendering and backward computation of Odin: Primitive-Level
Synchronization for Distributed Point-Based Neural Rendering, Figure 7): gs_preprocess,
gs_bin_and_sort, gs_render_fwd, gs_render_bwd_sqerr, gs_preprocess_bwd. The loss is the squared
error 0.5 |image - target|^2; its gradient dL/dimage = image - target is formed by the backward
kernel itself as it reads the image (gs_render_bwd_sqerr), so every kernel of the step is the
library's. A caller with its own loss passes its dL/dimage (`upstream`) to gs_render_bwd instead.
Parameter gradients of the views of one step are summed (the first view overwrites, the others
accumulate).
"""
from __future__ import annotations

import torch

from . import api


class StepBuffers:
    """Device buffers reused across steps for scenes of a fixed size."""

    def __init__(self, n: int, device):
        self.device = torch.device(device)
        self.proj = api.alloc_proj(n, self.device)
        self.sort = api.SortBuffers(self.device)
        self.grad2d = torch.empty((n, 12), dtype=torch.float32, device=self.device)
        self.images = {}
        self.n = n
        self._surfel = None

    def surfel_buffers(self):
        """(rec2d [N, 16], grad2d [N, 16]) of the surfel pipeline, allocated on first use."""
        if self._surfel is None:
            self._surfel = (torch.empty((self.n, 16), dtype=torch.float32, device=self.device),
                            torch.empty((self.n, 16), dtype=torch.float32, device=self.device))
        return self._surfel

    def image_buffers(self, width: int, height: int):
        key = (width, height)
        if key not in self.images:
            d = self.device
            self.images[key] = (torch.empty((3, height, width), dtype=torch.float32, device=d),
                                torch.empty((height, width), dtype=torch.float32, device=d),
                                torch.empty((height, width), dtype=torch.int32, device=d),
                                torch.empty((3, height, width), dtype=torch.float32, device=d),
                                torch.empty((((height + 15) // 16) * ((width + 15) // 16), 2), dtype=torch.int32,
                                            device=d))
        return self.images[key]


def train_step(params: dict, cameras, targets, opt, grads: dict, buffers: StepBuffers, capacity: int | None = None,
               want_keys: bool = False, stream=None) -> dict:
    """Runs every view and leaves the summed parameter gradients in `grads`. Returns per-view
    duplicate counts and the last view's image (a view of a reused buffer)."""
    n_dups = []
    image = None
    for v, (cam, target) in enumerate(zip(cameras, targets)):
        c = api.make_camera(cam)
        proj = api.gs_preprocess(params, c, opt, out=buffers.proj, stream=stream)
        image, t_final, n_contrib, dl, ranges = buffers.image_buffers(c.width, c.height)
        b = api.gs_bin_and_sort(proj, c, opt, capacity=capacity, buffers=buffers.sort, want_keys=want_keys,
                                ranges=ranges, stream=stream)
        api.gs_render_fwd(proj, b.vals, b.ranges, c, opt, out=(image, t_final, n_contrib), stream=stream)
        api.gs_render_bwd_sqerr(proj, b.vals, b.ranges, c, opt, image, target, t_final, n_contrib,
                                grad2d=buffers.grad2d, stream=stream)
        api.gs_preprocess_bwd(params, c, opt, proj, buffers.grad2d, out=grads, accumulate=v > 0, stream=stream)
        n_dups.append(b.n_dup)
    return {"n_dup": n_dups, "image": image}


def train_step_async(params: dict, cameras, targets, opt, grads: dict, buffers: StepBuffers, capacity: int,
                     n_dup: torch.Tensor, events=None, stream=None, upstream=None, losses=None):
    """train_step without any host synchronisation: the sort is gs_bin_and_sort_async with a
    fixed capacity, and the views' duplicate counts land in the device tensor n_dup [views]
    (a view whose count exceeds the capacity renders nothing and sets the device check error).
    events: optional per view ((fwd start, fwd end), (bwd start, bwd end)) recorded around the
    two raster kernels (on the current stream). upstream: optional per-view dL/dimage [3, H, W]
    tensors supplied by the caller (a loss computed elsewhere); the targets are then unused.
    losses: optional device float tensor [views] receiving each view's squared-error loss."""
    image = None
    for v, (cam, target) in enumerate(zip(cameras, targets)):
        ev = events[v] if events is not None else None
        c = cam if isinstance(cam, api.gs_camera) else api.make_camera(cam)
        proj = api.gs_preprocess(params, c, opt, out=buffers.proj, stream=stream)
        image, t_final, n_contrib, dl, ranges = buffers.image_buffers(c.width, c.height)
        b = api.gs_bin_and_sort_async(proj, c, opt, capacity, buffers=buffers.sort, ranges=ranges,
                                      n_dup=n_dup[v:v + 1], stream=stream)
        if ev is not None:
            ev[0][0].record()
        api.gs_render_fwd(proj, b.vals, b.ranges, c, opt, out=(image, t_final, n_contrib), stream=stream)
        if ev is not None:
            ev[0][1].record()
            ev[1][0].record()
        if upstream is None:
            api.gs_render_bwd_sqerr(proj, b.vals, b.ranges, c, opt, image, target, t_final, n_contrib,
                                    grad2d=buffers.grad2d, loss=losses[v:v + 1] if losses is not None else None,
                                    stream=stream)
        else:
            api.gs_render_bwd(proj, b.vals, b.ranges, c, opt, upstream[v], t_final, n_contrib,
                              grad2d=buffers.grad2d, stream=stream)
        if ev is not None:
            ev[1][1].record()
        api.gs_preprocess_bwd(params, c, opt, proj, buffers.grad2d, out=grads, accumulate=v > 0, stream=stream)
    return image


def train_step_async_overlapped(params: dict, cameras, targets, opt, grads: dict, buffers, capacity: int,
                                n_dup: torch.Tensor, events=None, upstream=None, losses=None, streams=None):
    """train_step_async for several views with two buffer sets (`buffers`: two StepBuffers) on two
    streams: view v runs on stream v % 2 with buffer set v % 2, so that one view's preprocess, sort
    and rasterization overlap the other's. The preprocess backward of view v waits for view v - 1's,
    so the views' gradients are added in view order as in train_step_async; a buffer set is reused
    two views later, after its stream has finished with it. Both streams fork from and join the
    current stream (so the step can be captured into a CUDA graph from it). streams: the two side
    streams (created here when None)."""
    main = torch.cuda.current_stream()
    if streams is None:
        streams = [torch.cuda.Stream(main.device), torch.cuda.Stream(main.device)]
    for st in streams:
        st.wait_stream(main)
    prev = None  # event after the previous view's preprocess backward
    image = None
    for v, (cam, target) in enumerate(zip(cameras, targets)):
        st, buf = streams[v % 2], buffers[v % 2]
        ev = events[v] if events is not None else None
        c = cam if isinstance(cam, api.gs_camera) else api.make_camera(cam)
        with torch.cuda.stream(st):
            proj = api.gs_preprocess(params, c, opt, out=buf.proj, stream=st)
            image, t_final, n_contrib, dl, ranges = buf.image_buffers(c.width, c.height)
            b = api.gs_bin_and_sort_async(proj, c, opt, capacity, buffers=buf.sort, ranges=ranges,
                                          n_dup=n_dup[v:v + 1], stream=st)
            if ev is not None:
                ev[0][0].record(st)
            api.gs_render_fwd(proj, b.vals, b.ranges, c, opt, out=(image, t_final, n_contrib), stream=st)
            if ev is not None:
                ev[0][1].record(st)
                ev[1][0].record(st)
            if upstream is None:
                api.gs_render_bwd_sqerr(proj, b.vals, b.ranges, c, opt, image, target, t_final, n_contrib,
                                        grad2d=buf.grad2d, loss=losses[v:v + 1] if losses is not None else None,
                                        stream=st)
            else:
                api.gs_render_bwd(proj, b.vals, b.ranges, c, opt, upstream[v], t_final, n_contrib,
                                  grad2d=buf.grad2d, stream=st)
            if ev is not None:
                ev[1][1].record(st)
            if prev is not None:
                st.wait_event(prev)
            api.gs_preprocess_bwd(params, c, opt, proj, buf.grad2d, out=grads, accumulate=v > 0, stream=st)
            prev = torch.cuda.Event()
            prev.record(st)
    for st in streams:
        main.wait_stream(st)
    return image


def train_step_surfels_async(params: dict, cameras, targets, opt, grads: dict, buffers: StepBuffers, capacity: int,
                             n_dup: torch.Tensor, events=None, stream=None):
    """train_step_async for the surfel (2D Gaussian splatting) pipeline: gs_preprocess2d, the same
    sort, gs_render2d_fwd, the loss gradient, gs_render2d_bwd, gs_preprocess2d_bwd."""
    rec2d, g2d = buffers.surfel_buffers()
    image = None
    for v, (cam, target) in enumerate(zip(cameras, targets)):
        ev = events[v] if events is not None else None
        c = cam if isinstance(cam, api.gs_camera) else api.make_camera(cam)
        proj, _ = api.gs_preprocess2d(params, c, opt, out=buffers.proj, rec2d=rec2d, stream=stream)
        image, t_final, n_contrib, dl, ranges = buffers.image_buffers(c.width, c.height)
        b = api.gs_bin_and_sort_async(proj, c, opt, capacity, buffers=buffers.sort, ranges=ranges,
                                      n_dup=n_dup[v:v + 1], stream=stream)
        if ev is not None:
            ev[0][0].record()
        api.gs_render2d_fwd(rec2d, b.vals, b.ranges, c, opt, out=(image, t_final, n_contrib), stream=stream)
        if ev is not None:
            ev[0][1].record()
        torch.sub(image, target, out=dl)
        if ev is not None:
            ev[1][0].record()
        api.gs_render2d_bwd(rec2d, b.vals, b.ranges, c, opt, dl, t_final, n_contrib, grad2d=g2d, stream=stream)
        if ev is not None:
            ev[1][1].record()
        api.gs_preprocess2d_bwd(params, c, opt, proj, g2d, out=grads, accumulate=v > 0, stream=stream)
    return image


class GraphedStep:
    """The step of fixed views (train_step_async) captured into one CUDA graph: replay() runs
    every kernel of the step with one launch from the host. Inputs are read from, and gradients
    written to, the same tensors at every replay (update them in place between replays)."""

    def __init__(self, params: dict, cameras, targets, opt, grads: dict, buffers: StepBuffers, capacity: int,
                 events=None, surfels: bool = False, upstream=None, buffers2: StepBuffers | None = None):
        """events: as for train_step_async; to time kernels inside the graph they must be created
        with torch.cuda.Event(enable_timing=True, external=True), which captures them as event
        record nodes. surfels: capture the surfel pipeline (train_step_surfels_async) instead.
        upstream: per-view dL/dimage tensors read at every replay instead of image - target
        (3D pipeline only). buffers2: a second buffer set; with it and several views the 3D
        pipeline runs its views on two streams (train_step_async_overlapped)."""
        self.device = buffers.device
        self.cams = [c if isinstance(c, api.gs_camera) else api.make_camera(c) for c in cameras]
        self.n_dup = torch.zeros(len(self.cams), dtype=torch.int64, device=self.device)
        self.losses = torch.zeros(len(self.cams), dtype=torch.float32, device=self.device)  # per view (3D pipeline)
        args = (params, self.cams, targets, opt, grads, buffers, capacity, self.n_dup, events)
        if surfels:
            assert upstream is None, "upstream gradients are supported by the 3D pipeline only"
            run = train_step_surfels_async
        elif buffers2 is not None and len(self.cams) > 1:
            side_streams = [torch.cuda.Stream(self.device), torch.cuda.Stream(self.device)]

            def run(p, cams, tg, o, g, bufs, cap, nd, ev):
                return train_step_async_overlapped(p, cams, tg, o, g, [bufs, buffers2], cap, nd, events=ev,
                                                   upstream=upstream,
                                                   losses=None if upstream is not None else self.losses,
                                                   streams=side_streams)
        else:
            def run(*a):
                return train_step_async(*a, upstream=upstream, losses=None if upstream is not None else self.losses)
        # one eager run first: buffers, function attributes and device symbols are set up outside the capture
        side = torch.cuda.Stream(self.device)
        side.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(side):
            run(*args)
        torch.cuda.current_stream(self.device).wait_stream(side)
        torch.cuda.synchronize(self.device)
        before = api.gs_kernel_launches()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            run(*args)
        self.launches = api.gs_kernel_launches() - before  # library kernels per replay

    def replay(self):
        self.graph.replay()
