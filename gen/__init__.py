"""Seeded synthetic inputs shared by the CPU oracle and the GPU path (no method arithmetic)."""
