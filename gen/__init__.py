"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the bench."""
from .scenes import Scene, edge_scene, lego_scene, look_at_camera, random_scene
from .workloads import (CONFIGS, SPLAT_FIELDS, Workload, elongated_fixture, from_arrays, lego_early, random_case,
                        lego_far, lego_final, make, overlap_fixture, small, stress, tiny)

__all__ = ["Scene", "edge_scene", "lego_scene", "look_at_camera", "random_scene", "CONFIGS", "SPLAT_FIELDS", "Workload", "from_arrays", "make", "overlap_fixture",
           "elongated_fixture", "random_case", "tiny", "small", "lego_early", "lego_final", "lego_far", "stress"]
