"""B300-native DCNv3/DCNv4 core deformable aggregation (placeholder, binding follows)."""
