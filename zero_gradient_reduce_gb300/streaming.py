"""ZeRO-2 streaming of one step through zdp_step, overlapped with the producer
of the gradients.

CS336 Lecture 7 notes, 8.2 (ZeRO-2), items 1-4: as the backward pass produces
each layer's gradients they are reduce-scattered right away and freed, and
every rank updates the shard it owns; 6.4 gives the reason to work in buckets
(fewer, larger messages, overlapped with the backward pass).  Here the P ranks
share one GPU, the "backward pass" is whatever the caller's `produce` callback
enqueues, and each bucket of the flat model is handed to zdp_step with
off/len as soon as it is written.

Two CUDA streams and two events per bucket order the work:
  - the producer stream writes bucket b's P gradient slices into one of
    `buffers` bucket buffers (double-buffered by default) and records
    ready[b];
  - the step stream waits for ready[b], runs zdp_step on bucket b and records
    done[b];
  - before the producer reuses a buffer for bucket b + buffers it waits for
    done[b].
So the producer fills bucket b+1 while the step runs on bucket b.  Ownership
in zdp_step is global (it depends only on the element's index and n), so the
streamed step gives the same bits as one call over the whole model.

This module is host-side orchestration only: it allocates the bucket buffers
with torch and enqueues zdp_step calls; every step of the computation runs in
libzdp's kernels.
"""

from __future__ import annotations

from typing import Callable, List, Optional, Sequence, Tuple

import torch

from . import zdp


def bucket_bounds(n: int, bucket_elems: int) -> List[Tuple[int, int]]:
    """[lo, hi) of each bucket of a flat model of n elements (the last one
    ragged)."""
    if n < 1 or bucket_elems < 1:
        raise ValueError(f"n={n} and bucket_elems={bucket_elems} must be >= 1")
    return [(lo, min(n, lo + bucket_elems)) for lo in range(0, n, bucket_elems)]


class StepTimes:
    """CUDA events of one streamed step: start (on the caller's stream) and
    end (after the last zdp_step), and each zdp_step's own start and end on
    the step stream.  Read them after the step has completed."""

    def __init__(self, nbuckets: int):
        def ev():
            return torch.cuda.Event(enable_timing=True)
        self.start, self.end = ev(), ev()
        self.step0 = [ev() for _ in range(nbuckets)]
        self.step1 = [ev() for _ in range(nbuckets)]

    def wall_ms(self) -> float:
        """From the call's start to the last bucket's update."""
        return self.start.elapsed_time(self.end)

    def step_ms(self) -> float:
        """Sum of the zdp_step launches' own durations."""
        return sum(a.elapsed_time(b) for a, b in zip(self.step0, self.step1))


class StreamedStep:
    """One ZeRO step streamed through zdp_step bucket by bucket, with the
    gradient producer on its own stream.

    master/m/v/replicas, d_overflow and d_sumsq are as for zdp_step (whole
    model, global indices).  The object allocates `buffers` sets of P bucket
    buffers of `bucket_elems` gradients each, and builds one zdp_step_args per
    bucket.
    """

    def __init__(self, P: int, n: int, bucket_elems: int, master, m, v, replicas: Sequence,
                 *, scale: float, lr: float, b1: float, b2: float, eps: float, wd: float,
                 grad_dtype=torch.bfloat16, moments: str = "f32", d_overflow=None,
                 d_sumsq=None, buffers: int = 2, device=None):
        if buffers < 1:
            raise ValueError("at least one bucket buffer is needed")
        if len(replicas) != P:
            raise ValueError(f"{len(replicas)} replicas for P={P}")
        device = torch.device("cuda") if device is None else torch.device(device)
        self.P, self.n = P, n
        self.bounds = bucket_bounds(n, bucket_elems)
        B = min(bucket_elems, n)
        self.bufs = [[torch.empty(B, dtype=grad_dtype, device=device) for _ in range(P)]
                     for _ in range(buffers)]
        self.args = []
        for b, (lo, hi) in enumerate(self.bounds):
            views = [x[:hi - lo] for x in self.bufs[b % buffers]]
            self.args.append(zdp.make_step_args(
                views, master, m, v, replicas, n=n, scale=scale, lr=lr, b1=b1, b2=b2, eps=eps,
                wd=wd, t=1, off=lo, length=hi - lo, d_overflow=d_overflow, d_sumsq=d_sumsq,
                moments=moments))
        self.producer = torch.cuda.Stream(device)
        self.stepper = torch.cuda.Stream(device)
        # The buffers live on the two side streams: when they are freed, the
        # caching allocator must wait for the work queued there, not only for
        # the stream they were allocated on.
        for bufset in self.bufs:
            for x in bufset:
                x.record_stream(self.producer)
                x.record_stream(self.stepper)
        self.ready = [torch.cuda.Event() for _ in self.bounds]
        self.done = [torch.cuda.Event() for _ in self.bounds]

    def views(self, b: int) -> List[torch.Tensor]:
        """The P gradient slices bucket b is written into."""
        lo, hi = self.bounds[b]
        return [x[:hi - lo] for x in self.bufs[b % len(self.bufs)]]

    def run(self, t: int, produce: Callable[[List[torch.Tensor], int, int], None],
            times: Optional[StepTimes] = None) -> None:
        """Enqueues one step at AdamW step t.  produce(views, lo, hi) must
        enqueue, on the current stream (the producer's when it is called), the
        writes of rank q's gradients of elements [lo, hi) into views[q].

        The call is ordered like a launch on the caller's current stream: both
        streams first wait for the work already there (e.g. a reset of the
        flag words), and that stream waits for the last bucket's update."""
        caller = torch.cuda.current_stream()
        if times is not None:
            times.start.record(caller)
        self.producer.wait_stream(caller)
        self.stepper.wait_stream(caller)
        nbuf = len(self.bufs)
        for b, (lo, hi) in enumerate(self.bounds):
            with torch.cuda.stream(self.producer):
                if b >= nbuf:
                    self.producer.wait_event(self.done[b - nbuf])  # buffer free again
                produce(self.views(b), lo, hi)
                self.ready[b].record(self.producer)
            self.stepper.wait_event(self.ready[b])
            a = self.args[b][0]
            a.t = t
            if times is not None:
                times.step0[b].record(self.stepper)
            zdp.zdp_step(a, self.stepper)
            if times is not None:
                times.step1[b].record(self.stepper)
            self.done[b].record(self.stepper)
        if times is not None:
            times.end.record(self.stepper)
        caller.wait_stream(self.stepper)
        # the producer's last writes are ordered before the caller's next work too
        caller.wait_stream(self.producer)
